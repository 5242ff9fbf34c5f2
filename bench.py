"""Benchmark of the grouped-conv weight gradient on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-extra]

A step is one call of wg_conv_bwd_weight -- the whole path: every launch it makes
(split-K stage 1, the stage-2 reduce or the atomic-mode memset) -- over one batch
of synthetic, seeded inputs already resident in HBM.  The device-side value
times the K steps back to back between one pair of CUDA events on the calls'
stream and divides by K (steps that need an L2 flush are timed one by one, the
flush outside the events; --graph replays a captured CUDA graph of the call
instead).  The e2e value times wg_conv_bwd_weight_host,
the same computation from pinned host buffers: X and dY copied in, the call,
dW copied back, all enqueued by the library.  The headline workload is the 2-D dense 56x56, C = K = 64, N = 32, 3x3
problem with bf16 inputs and bf16 dW; the other workloads, and the other plans
the measurement table lists for each (split degrees, modes, merge widths, the
tensor-core depthwise variant, the tensor-core kernel with every filter tap on
the MMA rows), are reported under "workloads".  No step finds
its inputs in L2: each step reads the next of several copies of X and dY whose
total exceeds twice the L2; inputs too small for that (the 8x8 problem) are
evicted instead by an L2 flush before every step (a 256 MiB write, then a
256 MiB read of another buffer so the write's dirty lines are written back
before the timed events).  The roofline's kernel time comes from a second pass
over the same steps with an event recorded at each step's start and one right
after its main kernel.

Prints one JSON line on rank 0.  Multi-GPU runs (torchrun) are independent
replicas (weak scaling): the path has no exchange step on one node.
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

from implicit_gemm_gb300 import binding, build, synth  # noqa: E402

L2_FLUSH_BYTES = 256 << 20


def spec(ndim, G, N, C, K, inn, filt, stride, dil, pl, pr, in_dtype, out_dtype):
    return {"ndim": ndim, "G": G, "N": N, "C": C, "K": K, "in": inn, "filt": filt, "stride": stride, "dil": dil,
            "pad_l": pl, "pad_r": pr, "in_dtype": in_dtype, "out_dtype": out_dtype}


# name -> (spec, distribution, seed index, split_k, mode, group_merge)
WORKLOADS = {
    "2d_dense_n32_h56_c64_k64": (spec(2, 1, 32, 64, 64, [56, 56], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], "bf16",
                                      "bf16"), ("uniform", -1.0, 1.0), 2, 0, "auto", 0),
    "2d_tiny_n1_h8_c16_k32": (spec(2, 1, 1, 16, 32, [8, 8], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], "bf16", "fp32"),
                              ("uniform", -1.0, 1.0), 1, 0, "auto", 0),
    "2d_grouped_g32_c8_k8_n32_h28": (spec(2, 32, 32, 8, 8, [28, 28], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], "bf16",
                                          "fp32"), ("normal", 0.0, 1.0), 3, 0, "auto", 0),
    "2d_depthwise_g512_n64_h28": (spec(2, 512, 64, 1, 1, [28, 28], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], "bf16",
                                       "fp32"), ("uniform", -1.0, 1.0), 4, 0, "auto", 0),
    "3d_n4_d16_c128_k96_s2": (spec(3, 1, 4, 128, 96, [16, 16, 16], [3, 3, 3], [2, 2, 2], [1, 1, 1], [1, 1, 1],
                                   [1, 1, 1], "fp16", "fp32"), ("normal", 0.0, 0.5), 5, 8, "atomic", 0),
}
WORKLOADS["2d_1x1_n32_h56_c64_k256"] = (spec(2, 1, 32, 64, 256, [56, 56], [1, 1], [1, 1], [1, 1], [0, 0], [0, 0],
                                             "bf16", "fp32"), ("uniform", -1.0, 1.0), 6, 0, "auto", 0)
WORKLOADS["2d_1x1s2_n32_h56_c256_k128"] = (spec(2, 1, 32, 256, 128, [56, 56], [1, 1], [2, 2], [1, 1], [0, 0], [0, 0],
                                                "bf16", "fp32"), ("uniform", -1.0, 1.0), 7, 0, "auto", 0)
HEADLINE = "2d_dense_n32_h56_c64_k64"

# Plans reported under "workloads": (label, workload, split_k, mode, group_merge, kernel).
VARIANTS = [
    ("2d_tiny_n1_h8_c16_k32", "2d_tiny_n1_h8_c16_k32", 0, "auto", 0, "auto"),
    ("2d_dense_n32_h56_c64_k64/S1_direct", "2d_dense_n32_h56_c64_k64", 1, "direct", 0, "auto"),
    ("2d_dense_n32_h56_c64_k64/S4_deterministic", "2d_dense_n32_h56_c64_k64", 4, "deterministic", 0, "auto"),
    ("2d_dense_n32_h56_c64_k64/taps_m", "2d_dense_n32_h56_c64_k64", 0, "auto", 0, "igemm_taps_m"),
    ("2d_grouped_g32_c8_k8_n32_h28", "2d_grouped_g32_c8_k8_n32_h28", 0, "auto", 0, "auto"),
    ("2d_grouped_g32_c8_k8_n32_h28/deterministic", "2d_grouped_g32_c8_k8_n32_h28", 0, "deterministic", 0, "auto"),
    # Merge degrees with the two-stage epilogue pinned, as the pages compare them.
    ("2d_depthwise_g512_n64_h28/gm8", "2d_depthwise_g512_n64_h28", 0, "deterministic", 8, "auto"),
    ("2d_depthwise_g512_n64_h28/gm1", "2d_depthwise_g512_n64_h28", 0, "deterministic", 1, "auto"),
    ("2d_depthwise_g512_n64_h28/gm2", "2d_depthwise_g512_n64_h28", 0, "deterministic", 2, "auto"),
    ("2d_depthwise_g512_n64_h28", "2d_depthwise_g512_n64_h28", 0, "auto", 0, "auto"),
    ("2d_depthwise_g512_n64_h28/gm4", "2d_depthwise_g512_n64_h28", 0, "deterministic", 4, "auto"),
    ("2d_depthwise_g512_n64_h28/gm4_atomic", "2d_depthwise_g512_n64_h28", 0, "atomic", 4, "auto"),
    ("2d_depthwise_g512_n64_h28/tensor_core", "2d_depthwise_g512_n64_h28", 0, "auto", 0, "igemm"),
    ("3d_n4_d16_c128_k96_s2", "3d_n4_d16_c128_k96_s2", 8, "atomic", 0, "auto"),
    ("3d_n4_d16_c128_k96_s2/S8_deterministic", "3d_n4_d16_c128_k96_s2", 8, "deterministic", 0, "auto"),
    ("3d_n4_d16_c128_k96_s2/auto", "3d_n4_d16_c128_k96_s2", 0, "auto", 0, "auto"),
    ("2d_1x1_n32_h56_c64_k256", "2d_1x1_n32_h56_c64_k256", 0, "auto", 0, "auto"),
    ("2d_1x1s2_n32_h56_c256_k128", "2d_1x1s2_n32_h56_c256_k128", 0, "auto", 0, "auto"),
]


def out_dims(sp):
    return binding.wg_problem_normalize(sp)


def sizes(sp, dims=None):
    """Element counts, FLOPs and algorithmic bytes of a problem.  `dims` computes the
    output lengths (the library's normalisation by default; the reference arm passes
    the oracle's, so that it never loads the library)."""
    o = (dims or out_dims)(sp)
    T = int(np.prod(sp["filt"]))
    P = sp["N"] * int(np.prod(o))
    nx = sp["N"] * int(np.prod(sp["in"])) * sp["G"] * sp["C"]
    ndy = P * sp["G"] * sp["K"]
    ndw = sp["G"] * sp["K"] * T * sp["C"]
    flops = 2.0 * sp["G"] * sp["K"] * sp["C"] * T * P
    wsz = 4 if sp["out_dtype"] == "fp32" else 2
    return {"out": o, "nx": nx, "ndy": ndy, "ndw": ndw, "flops": flops,
            "bytes": 2.0 * nx + 2.0 * ndy + float(wsz) * ndw, "wsz": wsz}


# The five configurations and the modes each is quoted in, as VARIANTS labels
# (the main line's label is its workload name), for the compact per-config
# summary printed at the end of the JSON line.
CONFIG_LABELS = [
    ("c1_tiny", "2d_tiny_n1_h8_c16_k32"),
    ("c2_dense_auto", "2d_dense_n32_h56_c64_k64"),
    ("c2_dense_S1_direct", "2d_dense_n32_h56_c64_k64/S1_direct"),
    ("c2_dense_S4_det", "2d_dense_n32_h56_c64_k64/S4_deterministic"),
    ("c3_grouped_auto", "2d_grouped_g32_c8_k8_n32_h28"),
    ("c3_grouped_det", "2d_grouped_g32_c8_k8_n32_h28/deterministic"),
    ("c4_dw_auto", "2d_depthwise_g512_n64_h28"),
    ("c4_dw_gm1", "2d_depthwise_g512_n64_h28/gm1"),
    ("c4_dw_gm2", "2d_depthwise_g512_n64_h28/gm2"),
    ("c4_dw_gm4", "2d_depthwise_g512_n64_h28/gm4"),
    ("c4_dw_gm8", "2d_depthwise_g512_n64_h28/gm8"),
    ("c4_dw_gm4_atomic", "2d_depthwise_g512_n64_h28/gm4_atomic"),
    ("c4_dw_tensor_core", "2d_depthwise_g512_n64_h28/tensor_core"),
    ("c5_3d_S8_atomic", "3d_n4_d16_c128_k96_s2"),
    ("c5_3d_S8_det", "3d_n4_d16_c128_k96_s2/S8_deterministic"),
    ("c5_3d_auto", "3d_n4_d16_c128_k96_s2/auto"),
]


def plan_tag(plan):
    """A few words of a plan string: kernel, tile form, mode, split degree, merge width."""
    f = dict(kv.split("=", 1) for kv in plan.split() if "=" in kv)
    if f.get("kernel") == "depthwise":
        return f"dw Gm{f['Gm']} {f['mode'][:3]} S{f['S']}"
    pair = " pair" if f.get("code") == "pair" else ""
    return f"tc {f.get('taps', '')}{pair} {f['mode'][:3]} S{f['S']} Gm{f.get('Gm', 1)}"


def compact_configs(main_label, main, extra):
    """Per configuration: [step us, main-kernel roofline fraction, step roofline fraction, plan tag]."""
    out = {"fields": ["step_us", "kernel_frac", "step_frac", "plan"]}
    for key, label in CONFIG_LABELS:
        r = main if label == main_label else extra.get(label)
        if r is None:
            continue
        out[key] = [round(r["ms_per_step"] * 1e3, 2), round(r["kernel_roofline_frac"], 3),
                    round(r["roofline_frac"], 3), r["tag"]]
    return out


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return {"hbm": float(d["hbm_gbs"]), "bf16": float(d["bf16_tflops"]),
                "bf16_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "src": "measured"}
    except Exception:
        return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "src": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(dist, ms, device):
    """The slowest rank's time (ms): every rank gets the same value.  `dist` is
    torch.distributed with an initialised process group (NCCL on the GPUs; the
    tests use gloo on the CPU), or None for a single process."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world_size, units_per_rank, ms):
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return world_size * units_per_rank / (ms * 1e-3)


def run_reference(args, ws, rank):
    """Reference arm: the fp64 CPU oracle, as it stands, on this host's cores."""
    import oracle  # the one other place the bench runs the oracle
    if rank != 0:
        return
    sp = dict(WORKLOADS[args.workload][0])
    # A bounded sample of the workload: one of the batch's images per step.
    nsample = 1
    sps = dict(sp, N=nsample)
    dist, seed = WORKLOADS[args.workload][1], WORKLOADS[args.workload][2]
    s = sizes(sps, oracle.out_dims)
    x = oracle.decode(synth.tensor_bits(1000 + seed, s["nx"], sp["in_dtype"], *dist), sp["in_dtype"])
    dy = oracle.decode(synth.tensor_bits(2000 + seed, s["ndy"], sp["in_dtype"], *dist), sp["in_dtype"])
    for _ in range(args.warmup):
        oracle.wgrad(sps, x, dy)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.wgrad(sps, x, dy)
    dt = (time.perf_counter() - t0) / args.steps
    value = s["flops"] / dt / 1e12
    line = {"impl": "reference", "metric": "wgrad TFLOP/s", "value": value, "unit": "TFLOP/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": args.workload, "sample_images": nsample},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.threads(), "kind": "oracle",
                             "sample": f"{nsample} of {sp['N']} images of {args.workload} per step"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline(name):
    """The oracle timed on this host's cores on the full workload: whole runs until about
    10 s of CPU work have been timed."""
    import oracle
    sp, dist, seed = WORKLOADS[name][0], WORKLOADS[name][1], WORKLOADS[name][2]
    s = sizes(sp, oracle.out_dims)
    x = oracle.decode(synth.tensor_bits(1000 + seed, s["nx"], sp["in_dtype"], *dist), sp["in_dtype"])
    dy = oracle.decode(synth.tensor_bits(2000 + seed, s["ndy"], sp["in_dtype"], *dist), sp["in_dtype"])
    runs, t0 = 0, time.perf_counter()
    while runs < 1 or time.perf_counter() - t0 < 10.0:
        oracle.wgrad(sp, x, dy)
        runs += 1
    dt = (time.perf_counter() - t0) / runs
    return {"value": s["flops"] / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.threads(), "kind": "oracle",
            "sample": f"full {name} workload, {runs} run(s), fp64 direct loop with |dY*X| sums"}


L2_BYTES = 129 * 1000 * 1000
# DRAM bytes (read + write) of one launch of the main kernel of a plan (a
# VARIANTS label, or a workload name for its default plan) from an ncu capture
# of the kernel as it now stands (summaries under profiles/); a plan without
# such a capture reports null.  ncu flushes the caches before the captured
# launch, so atomic plans also count the dW lines their atomic adds fetch.
TRAFFIC = {
    # igemm_wgrad_kernel<1> (x taps on the columns, one M-tile), S = 75 two-stage: 25,776,384 B read + 0 B written.
    "2d_dense_n32_h56_c64_k64": 25_776_384,
    # igemm_wgrad_pair_kernel (CTA pairs), S = 4 two-stage: 25,751,552 B read + 0 B written.
    "2d_dense_n32_h56_c64_k64/S4_deterministic": 25_751_552,
    # igemm_wgrad_kernel<0>, Gm = 8 fold, 32 x 4 pixel tiles, staged atomic output: 25,854,720 B read + 0 B written.
    "2d_grouped_g32_c8_k8_n32_h28": 25_854_720,
    # depthwise_wgrad_kernel<bf16, 2, sliding>, atomic: 103,135,744 B read + 3,367,680 B written.
    "2d_depthwise_g512_n64_h28": 106_503_424,
    # igemm_wgrad_kernel<0>, per-tap S = 8 atomic (two 128-pixel K-tiles per split): 6,015,744 B read + 0 B written.
    "3d_n4_d16_c128_k96_s2": 6_015_744,
    # igemm_wgrad_kernel<0>, per-tap S = 4 atomic: 6,010,624 B read (X + dY + the dW lines) + 0 B written.
    "3d_n4_d16_c128_k96_s2/auto": 6_010_624,
    # igemm_wgrad_kernel<0>, S = 87 atomic: 64,386,304 B read + 308,480 B written.
    "2d_1x1_n32_h56_c64_k256": 64_694_784,
    # igemm_wgrad_kernel<0>, per-tap S = 49 atomic: 19,497,472 B read + 0 B written.
    "2d_1x1s2_n32_h56_c256_k128": 19_497_472,
}
MAX_COPIES = 512


class Workload:
    """One workload's inputs, outputs and prepared calls.

    So that no step finds its inputs in L2, each step reads the next of `copies`
    identical copies of X and dY whose total size exceeds twice the L2 (a copy
    was last read more than 129 MB of other input ago).  Inputs too small for
    that within MAX_COPIES fall back to flushing L2 before every step."""

    def __init__(self, torch, name, rotate=True, plan=None):
        self.torch = torch
        self.name = name
        sp, dist, seed, self.split_k, self.mode, self.gm = WORKLOADS[name]
        self.kernel = "auto"
        if plan is not None:
            self.split_k, self.mode, self.gm, self.kernel = plan
        self.sp = sp
        self.s = sizes(sp)
        tdt = torch.bfloat16 if sp["in_dtype"] == "bf16" else torch.float16
        xb = synth.tensor_bits(1000 + seed, self.s["nx"], sp["in_dtype"], *dist)
        dyb = synth.tensor_bits(2000 + seed, self.s["ndy"], sp["in_dtype"], *dist)
        self.x_host = torch.from_numpy(xb.view(np.int16)).view(tdt).pin_memory()
        self.dy_host = torch.from_numpy(dyb.view(np.int16)).view(tdt).pin_memory()
        self.x = self.x_host.cuda()
        self.dy = self.dy_host.cuda()
        odt = {"fp32": torch.float32, "bf16": torch.bfloat16, "fp16": torch.float16}[sp["out_dtype"]]
        self.dw = torch.empty(self.s["ndw"], dtype=odt, device="cuda")
        self.dw_host = torch.empty(self.s["ndw"], dtype=odt).pin_memory()
        kw = {"kernel": self.kernel}
        self.ws_bytes = binding.wg_workspace_size(sp, self.split_k, self.mode, self.gm, **kw)
        self.ws = torch.empty(max(self.ws_bytes, 16), dtype=torch.uint8, device="cuda")
        self.plan = binding.wg_plan_string(sp, self.split_k, self.mode, self.gm, **kw)
        # This library's kernels per call: the main kernel, plus the split reduction
        # kernel ("reduce=kernel") or the kernel that zeroes dW before atomic
        # accumulation ("zero=kernel") where the plan has one.
        self.launches_per_step = 1 + (1 if "reduce=kernel" in self.plan else 0) + (1 if "zero=kernel" in self.plan else 0)
        self.call = binding.PreparedCall(sp, self.x, self.dy, self.dw, self.split_k, self.mode, self.gm, self.ws,
                                         self.ws_bytes, **kw)
        self.graph = None
        in_bytes = 2 * (self.s["nx"] + self.s["ndy"])
        need = -(-2 * L2_BYTES // in_bytes)
        self.copies = max(2, need) if rotate and need <= MAX_COPIES else 1
        self.calls = [self.call]
        self.inputs = [(self.x, self.dy)]
        for _ in range(self.copies - 1):
            xc, dyc = self.x.clone(), self.dy.clone()
            self.inputs.append((xc, dyc))
            self.calls.append(binding.PreparedCall(sp, xc, dyc, self.dw, self.split_k, self.mode, self.gm, self.ws,
                                                   self.ws_bytes, **kw))
        self.next = 0
        self.rotating = self.copies > 1
        # End to end: the host-buffer entry point, staging into self.x / self.dy / self.dw.
        self.host_call = binding.PreparedHostCall(sp, self.x_host, self.dy_host, self.dw_host, self.x, self.dy,
                                                  self.dw, self.split_k, self.mode, self.gm, self.ws, self.ws_bytes,
                                                  **kw)

    def l2_note(self):
        if self.rotating:
            mb = self.copies * 2 * (self.s["nx"] + self.s["ndy"]) / 1e6
            return f"inputs rotate through {self.copies} copies ({mb:.0f} MB > 2x L2); no flush"
        return "flushed before every timed step (outside the events): write 256 MiB, then read another 256 MiB"

    def capture(self, stream):
        """Capture one step (every launch of the call) into a CUDA graph."""
        torch = self.torch
        with torch.cuda.stream(stream):
            self.call(stream.cuda_stream)  # first call: plan, tensor maps, kernel attributes
        stream.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=stream):
            self.call(stream.cuda_stream)
        stream.synchronize()

    def step(self, stream):
        if self.graph is not None:
            self.graph.replay()
        else:
            self.calls[self.next](stream.cuda_stream)
            self.next = (self.next + 1) % self.copies

    def e2e_step(self, stream):
        # One public call from host buffers: X and dY in, the computation, dW out.
        self.host_call(stream.cuda_stream)


class DgradWorkload:
    """Backward-data on a workload's geometry: dY and W resident (dY rotated through
    copies larger than 2x L2, like the weight-gradient inputs), dX written."""

    def __init__(self, torch, name):
        self.torch = torch
        sp, dist, seed = WORKLOADS[name][:3]
        self.sp = sp
        s = sizes(sp)
        tdt = torch.bfloat16 if sp["in_dtype"] == "bf16" else torch.float16
        odt = {"fp32": torch.float32, "bf16": torch.bfloat16, "fp16": torch.float16}[sp["out_dtype"]]
        dyb = synth.tensor_bits(2000 + seed, s["ndy"], sp["in_dtype"], *dist)
        wb = synth.tensor_bits(3000 + seed, s["ndw"], sp["in_dtype"], *dist)
        self.dy = torch.from_numpy(dyb.view(np.int16)).view(tdt).cuda()
        self.w = torch.from_numpy(wb.view(np.int16)).view(tdt).cuda()
        self.dx = torch.empty(s["nx"], dtype=odt, device="cuda")
        self.flops = s["flops"]
        self.bytes = 2 * (s["ndy"] + s["ndw"]) + s["nx"] * (4 if sp["out_dtype"] == "fp32" else 2)
        self.plan = binding.wg_bwd_data_plan_string(sp)
        need = -(-2 * L2_BYTES // (2 * s["ndy"]))
        self.copies = max(2, need) if need <= MAX_COPIES else 1
        self.dys = [self.dy] + [self.dy.clone() for _ in range(self.copies - 1)]
        nb = binding.wg_bwd_data_workspace_size(sp)
        self.ws = torch.empty(max(nb, 16), dtype=torch.uint8, device="cuda")
        self.calls = [binding.PreparedDgradCall(sp, d, self.w, self.dx, self.ws, nb) for d in self.dys]
        self.next = 0
        self.rotating = self.copies > 1
        self.graph = None

    def step(self, stream):
        self.calls[self.next](stream.cuda_stream)
        self.next = (self.next + 1) % self.copies


class L2Flush:
    """Evicts the inputs from L2 between timed steps: writes a 256 MiB buffer (twice
    the L2), then reads another 256 MiB buffer so that the write-back of the dirty
    lines the write leaves behind happens here and not inside the next timed step."""

    def __init__(self, torch):
        self.torch = torch
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        self.r = torch.ones(L2_FLUSH_BYTES // 8, dtype=torch.int64, device="cuda")
        self.sink = torch.empty((), dtype=torch.int64, device="cuda")

    def __call__(self):
        self.w.zero_()
        self.torch.sum(self.r, dim=0, out=self.sink)


def time_steps(torch, wl, steps, warmup, flush, stream, e2e=False, mark=False):
    """CUDA-event times (ms) of `steps` steps on `stream`, one entry per step;
    inputs not in L2 at each step (rotating copies, else an L2 flush before the
    step).  Steps that need no flush run back to back between one pair of events
    (every entry is then the average); flushed steps are timed one by one with
    the flush outside the events.  With `mark`, each time runs from the step's
    start to the end of the call's main kernel (an event the library records
    between its main and its reduction kernel)."""
    fn = wl.e2e_step if e2e else wl.step
    do_flush = not e2e and (not wl.rotating or wl.graph is not None)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            if do_flush:
                flush()
            fn(stream)
        stream.synchronize()
        if not do_flush and not mark:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(steps):
                fn(stream)
            b.record(stream)
            stream.synchronize()
            binding.wg_check_status(stream)
            return [a.elapsed_time(b) / steps] * steps
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        if mark:
            for _, b in evs:
                b.record(stream)  # creates the event before the library records it
            stream.synchronize()
        for a, b in evs:
            if do_flush:
                flush()
            a.record(stream)
            if mark:
                binding.wg_set_mark_event(b)
                fn(stream)
            else:
                fn(stream)
                b.record(stream)
        binding.wg_set_mark_event(None)
        stream.synchronize()
    binding.wg_check_status(stream)
    return [a.elapsed_time(b) for a, b in evs]


# Depthwise shapes for --sweep, in the style of the inverted-residual networks'
# depthwise layers (synthetic: the pages' 197-shape corpus is not available):
# (G, N, H = W, filter, stride).  5x5 filters exceed the CUDA-core kernel's 9
# taps and run on the tensor-core kernel.
SWEEP_SHAPES = [
    (32, 32, 112, 3, 1), (96, 32, 112, 3, 2), (144, 32, 56, 3, 1), (144, 32, 56, 3, 2), (192, 32, 28, 3, 1),
    (192, 32, 28, 3, 2), (384, 32, 14, 3, 1), (576, 32, 14, 3, 1), (576, 32, 14, 3, 2), (960, 32, 7, 3, 1),
    (512, 64, 28, 3, 1), (64, 16, 64, 3, 1), (240, 32, 28, 5, 1), (480, 32, 14, 5, 1), (672, 32, 14, 5, 2),
    (1152, 32, 7, 5, 1),
]


def run_sweep(torch, stream, flush, steps, warmup):
    """The automatic plan against fixed merge widths, modes and the tensor-core
    kernel on each shape.  Two comparisons: the automatic merge degree against
    Gm = 1 with the two-stage epilogue pinned (the pages' protocol), and the
    whole automatic plan against the fastest plan measured."""
    rows = []
    for i, (G, N, H, F, st) in enumerate(SWEEP_SHAPES):
        name = f"sweep_dw_g{G}_n{N}_h{H}_f{F}_s{st}"
        sp = spec(2, G, N, 1, 1, [H, H], [F, F], [st, st], [1, 1], [F // 2, F // 2], [F // 2, F // 2], "bf16", "fp32")
        WORKLOADS[name] = (sp, ("uniform", -1.0, 1.0), 100 + i, 0, "auto", 0)
        dw = F * F <= 9
        plans = [("auto", (0, "auto", 0, "auto")), ("auto_det", (0, "deterministic", 0, "auto"))]
        if dw:
            plans += [(f"gm{g}", (0, "auto", g, "depthwise")) for g in (1, 2, 4, 8)]
            plans += [(f"gm{g}_det", (0, "deterministic", g, "depthwise")) for g in (1, 2, 4, 8)]
        plans += [("tensor_core", (0, "auto", 0, "igemm")), ("tensor_core_det", (0, "deterministic", 0, "igemm"))]
        res = {}
        for label, plan in plans:
            try:
                wl = Workload(torch, name, plan=plan)
            except binding.WgradError:
                continue
            res[label] = float(np.mean(time_steps(torch, wl, steps, warmup, flush, stream))) * 1e3
            del wl
        best = min(res, key=res.get)
        row = {"shape": name, "auto_us": res["auto"], "best": best, "best_us": res[best],
               "auto_vs_best": res[best] / res["auto"], "plans_us": res,
               "auto_plan": plan_tag(binding.wg_plan_string(sp, 0, "auto", 0))}
        if "gm1_det" in res:
            row["auto_det_speedup_vs_gm1_det"] = res["gm1_det"] / res["auto_det"]
        rows.append(row)
        print(json.dumps(row), flush=True)
    gm = [r["auto_det_speedup_vs_gm1_det"] for r in rows if "auto_det_speedup_vs_gm1_det" in r]
    ab = [r["auto_vs_best"] for r in rows]
    geo = lambda v: float(np.exp(np.mean(np.log(v))))
    print(json.dumps({"sweep": "depthwise policy", "shapes": len(rows),
                      "geomean_auto_det_speedup_vs_gm1_det": geo(gm), "geomean_auto_vs_best": geo(ab),
                      "min_auto_vs_best": min(ab), "worst_shape": min(rows, key=lambda r: r["auto_vs_best"])["shape"]}),
          flush=True)


def run_floor(torch, flush, reps=20):
    """Cold-read floors, measured as the peaks in MEASURED_PEAKS.json are (torch ops,
    CUDA events) but with L2 flushed before each rep: for each workload's
    algorithmic bytes B, a copy of B/2 bytes (B of traffic) and a read-only
    reduction over B bytes; best and median of `reps` event-timed reps."""
    def timed(fn):
        ts = []
        for _ in range(reps + 3):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(); fn(); b.record(); torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) * 1e3)
        ts = ts[3:]
        return min(ts), statistics.median(ts)
    pk = peaks()
    for name in ("2d_dense_n32_h56_c64_k64", "2d_depthwise_g512_n64_h28", "3d_n4_d16_c128_k96_s2"):
        nbytes = int(sizes(WORKLOADS[name][0])["bytes"]) // 16 * 16
        a = torch.ones(nbytes // 4, dtype=torch.bfloat16, device="cuda")
        b = torch.empty_like(a)
        r = torch.ones(nbytes // 8, dtype=torch.int64, device="cuda")
        cp, cpm = timed(lambda: b.copy_(a))
        rd, rdm = timed(lambda: torch.sum(r))
        print(json.dumps({"floor": name, "bytes": nbytes, "copy_best_us": cp, "copy_median_us": cpm,
                          "read_best_us": rd, "read_median_us": rdm,
                          "copy_frac_of_peak": nbytes / (cp * 1e-6) / 1e9 / pk["hbm"],
                          "read_frac_of_peak": nbytes / (rd * 1e-6) / 1e9 / pk["hbm"]}), flush=True)
        del a, b, r


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE, choices=list(WORKLOADS))
    ap.add_argument("--variant", default=None, choices=[v[0] for v in VARIANTS],
                    help="time this listed plan (a label of VARIANTS) as the main line; sets --workload")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads and the CPU baseline")
    ap.add_argument("--graph", action="store_true", help="replay a CUDA graph of the call instead of calling it")
    ap.add_argument("--dgrad", action="store_true",
                    help="time backward-data on the workload's geometry instead of the weight gradient (no extras)")
    ap.add_argument("--floor", action="store_true",
                    help="time torch's copy and a read-only reduction of each workload's algorithmic bytes (cold L2)")
    ap.add_argument("--sweep", action="store_true",
                    help="time the automatic plan against fixed merge widths on a depthwise shape sweep")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return

    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device: the wgrad path has no CPU fallback")
    torch.cuda.set_device(local)
    pg = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist
    build.build()
    binding.load()
    stream = torch.cuda.Stream()
    flush = L2Flush(torch)
    pk = peaks()
    if args.floor:
        if rank == 0:
            run_floor(torch, flush)
        return
    if args.sweep:
        if rank == 0:
            run_sweep(torch, stream, flush, min(args.steps, 200), args.warmup)
        return
    if args.dgrad:
        w3 = DgradWorkload(torch, args.workload)
        ms = float(np.mean(time_steps(torch, w3, args.steps, args.warmup, flush, stream)))
        if rank == 0:
            print(json.dumps({"metric": "dgrad TFLOP/s", "value": w3.flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                              "ms_per_step": ms, "config": {"workload": args.workload, "plan": w3.plan}}), flush=True)
        return

    main_plan = None
    if args.variant:
        vlab = {v[0]: v for v in VARIANTS}[args.variant]
        args.workload, main_plan = vlab[1], tuple(vlab[2:])
    wl = Workload(torch, args.workload, plan=main_plan)
    if args.graph:
        wl.capture(stream)
    sampler = ClockSampler(local)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    t_wall = time.perf_counter()
    times = time_steps(torch, wl, args.steps, args.warmup, flush, stream)
    t_wall = time.perf_counter() - t_wall
    clocks = sampler.stop()
    torch.cuda.synchronize()
    step_ms = max_over_ranks(pg, float(np.mean(times)), "cuda")
    if pg:
        pg.barrier()
    s = wl.s
    value = job_value(ws, s["flops"], step_ms) / 1e12

    # End to end through the same C ABI call, host buffers: H2D of X and dY from
    # pinned memory, the call, D2H of dW, all inside the timed events.
    e2e_times = time_steps(torch, wl, max(20, args.steps // 10), args.warmup, flush, stream, e2e=True)
    e2e_ms = max_over_ranks(pg, float(np.mean(e2e_times)), "cuda")

    # Roofline of the dominant kernel (the call's main kernel: every FLOP of the
    # step and every algorithmic byte read or written goes through it): its
    # algorithmic FLOPs or bytes per launch over its average duration, measured
    # in a second pass over the same steps with an event the library records
    # right after it.  The bound is the slower of the two at the measured peaks.
    kern_ms = step_ms
    if not args.graph:
        kern_ms = float(np.mean(time_steps(torch, wl, args.steps, args.warmup, flush, stream, mark=True)))
    t_flop = s["flops"] / (pk["bf16"] * 1e12)
    t_byte = s["bytes"] / (pk["hbm"] * 1e9)
    if t_byte >= t_flop:
        roof = {"bound": "hbm", "achieved": s["bytes"] / (kern_ms * 1e-3) / 1e9, "peak": pk["hbm"], "unit": "GB/s"}
        roof["step_frac"] = s["bytes"] / (step_ms * 1e-3) / 1e9 / pk["hbm"]
    else:
        roof = {"bound": "tensor", "achieved": s["flops"] / (kern_ms * 1e-3) / 1e12, "peak": pk["bf16"],
                "unit": "TFLOP/s"}
        roof["step_frac"] = s["flops"] / (step_ms * 1e-3) / 1e12 / pk["bf16"]
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = TRAFFIC.get(args.variant or args.workload)
    roof["peak_source"] = pk["src"]
    roof["kernel"] = "igemm_wgrad_kernel" if "igemm" in wl.plan else "depthwise_wgrad_kernel"
    roof["kernel_ms"] = kern_ms
    roof["timed"] = ("main kernel: CUDA events from the step start to a mark the library records after the kernel"
                     if not args.graph else "whole step (graph replay) with CUDA events")

    extra = {}
    if rank == 0 and not args.no_extra:
        for label, name, *plan in VARIANTS:
            if label == (args.variant or args.workload):
                continue
            w2 = Workload(torch, name, plan=tuple(plan))
            if args.graph:
                w2.capture(stream)
            tt = time_steps(torch, w2, 300, 10, flush, stream)
            ms = float(np.mean(tt))
            kms = ms if args.graph else float(np.mean(time_steps(torch, w2, 300, 10, flush, stream, mark=True)))
            s2 = w2.s
            tf, tb = s2["flops"] / (pk["bf16"] * 1e12), s2["bytes"] / (pk["hbm"] * 1e9)
            extra[label] = {"ms_per_step": ms, "tflops": s2["flops"] / (ms * 1e-3) / 1e12,
                            "tag": plan_tag(w2.plan),
                           "gbs": s2["bytes"] / (ms * 1e-3) / 1e9, "roofline_us": max(tf, tb) * 1e6,
                           "bound": "hbm" if tb >= tf else "tensor",
                           "roofline_frac": max(tf, tb) / (ms * 1e-3), "kernel_ms": kms,
                           "kernel_roofline_frac": max(tf, tb) / (kms * 1e-3), "traffic": TRAFFIC.get(label),
                           "l2": w2.l2_note(), "plan": w2.plan}
            del w2
        # Backward-data (dgrad) on the dense and 1x1 geometries.
        for name in ("2d_dense_n32_h56_c64_k64", "2d_1x1_n32_h56_c64_k256"):
            w3 = DgradWorkload(torch, name)
            ms = float(np.mean(time_steps(torch, w3, 300, 10, flush, stream)))
            tf, tb = w3.flops / (pk["bf16"] * 1e12), w3.bytes / (pk["hbm"] * 1e9)
            extra["dgrad/" + name] = {"ms_per_step": ms, "tflops": w3.flops / (ms * 1e-3) / 1e12,
                                      "gbs": w3.bytes / (ms * 1e-3) / 1e9, "roofline_us": max(tf, tb) * 1e6,
                                      "bound": "hbm" if tb >= tf else "tensor",
                                      "roofline_frac": max(tf, tb) / (ms * 1e-3), "kernel_ms": ms,
                                      "kernel_roofline_frac": max(tf, tb) / (ms * 1e-3), "traffic": None,
                                      "l2": f"dY rotates through {w3.copies} copies", "plan": w3.plan}
            del w3

    if rank == 0:
        line = {"metric": "wgrad TFLOP/s", "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16" if wl.sp["in_dtype"] == "bf16" else "fp16",
                "data": "synthetic (seeded splitmix64)",
                "config": {"workload": args.workload, "variant": args.variant, "G": wl.sp["G"], "N": wl.sp["N"], "in": wl.sp["in"],
                           "C": wl.sp["C"], "K": wl.sp["K"], "filt": wl.sp["filt"], "stride": wl.sp["stride"],
                           "pad": wl.sp["pad_l"], "in_dtype": wl.sp["in_dtype"], "out_dtype": wl.sp["out_dtype"],
                           "split_k": wl.split_k, "mode": wl.mode, "plan": wl.plan,
                           "l2": wl.l2_note() if not args.graph else "flushed before every timed step (graph mode)",
                           "parallelism": f"replicas x{ws}"},
                "roofline": roof, "clocks": clocks, "gpu_launches": wl.launches_per_step * args.steps,
                "e2e": {"value": job_value(ws, s["flops"], e2e_ms) / 1e12, "unit": "TFLOP/s",
                        "h2d_bytes_per_step": 2 * (s["nx"] + s["ndy"]), "d2h_bytes_per_step": s["wsz"] * s["ndw"],
                        "ms_per_step": e2e_ms,
                        "call": "wg_conv_bwd_weight_host: pinned host X, dY in; dW out to pinned host memory"},
                "wall_s_timed": t_wall, "workloads": extra}
        if ws == 1 and not args.no_extra:
            line["cpu_baseline"] = cpu_baseline(args.workload)
        if extra:
            main = {"ms_per_step": step_ms, "kernel_roofline_frac": roof["frac"], "roofline_frac": roof["step_frac"],
                    "tag": plan_tag(wl.plan)}
            line["configs"] = compact_configs(args.variant or args.workload, main, extra)
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
