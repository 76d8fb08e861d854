#!/usr/bin/env python
"""Benchmark of the MoE layer forward with its aux-loss-free bias update on GB300.

One step = one moe_layer_fwd call over one batch of synthetic tokens: router, top-k,
gates, loads, stable permutation and gather, grouped routed-expert SwiGLU GEMMs,
shared-expert GEMMs, gated combine and the bias update (all in the library's CUDA
kernels).  Default workload: the Nano-shaped layer, T = 8192 tokens (batch 4 x
sequence 2048), d = 1024, 64 routed experts of width 512, top-2, shared width 2048.

Timing: W untimed warm-up steps, then K timed steps with a 512 MiB write between
steps (L2 is 129 MB, so every step starts cold), each step bracketed by CUDA events
on the launching stream; barrier + synchronize on both sides; max over ranks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload nano|skew|stack|tiny|train|...]
  python bench.py --impl reference ...   # the CPU oracle on the host cores

The `train` workload times a training step of the same layer instead: the forward
(saving its routing state) with the bias update, then moe_layer_bwd for a seeded
output gradient (dx and fp32 weight gradients of the router, routed and shared
experts).

Prints one JSON line.  Under torchrun (N > 1) every rank runs its own replica on its
own tokens (weak scaling); the only cross-rank exchange of the method is the sum of
the per-expert loads before the bias update.
"""
from __future__ import annotations

import argparse
import hashlib
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

from synth import (ATTN_CONFIGS, CONFIGS, f32_from_bf16_bits, make_attention, make_layer,  # noqa: E402
                   make_output_grad, make_tokens)

METRIC = "MoE-layer fwd tokens/s (T=8192,d=1024,64x512 top-2+2048 shared), % roofline"
FLUSH_BYTES = 512 << 20
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "gemm_chained_routed_ffn_nano_traffic.txt")
SHARED_TRAFFIC_FILE = os.path.join(ROOT, "profiles", "gemm_shared_gate_up_nano_traffic.txt")
TRAIN_TRAFFIC_FILE = os.path.join(ROOT, "profiles", "gemm_wgrad_gate_up_train_traffic.txt")
PROFILE_PERIOD = 10


def serve_step_roofline(fill_bytes, hbm_bytes, ms_step, link_gbs, peaks, peak_note):
    """The single-launch serving step (plan, fill and experts in one kernel): whichever
    of the host link (the step's fill bytes) and HBM (its weight bytes) bounds it."""
    link_s = fill_bytes / (link_gbs * 1e9) if link_gbs else 0.0
    hbm_s = hbm_bytes / (peaks["hbm_gbs"] * 1e9)
    if link_s > hbm_s:
        ach = fill_bytes / (ms_step / 1e3) / 1e9
        return {"kernel": "single-launch serving step (plan, fill from host memory, experts)", "bound": "link",
                "achieved": ach, "peak": link_gbs, "unit": "GB/s", "frac": ach / link_gbs, "traffic": None,
                "peak_note": "of a pinned host-to-device copy measured in this run"}
    ach = hbm_bytes / (ms_step / 1e3) / 1e9
    return {"kernel": "single-launch serving step (plan, fill from host memory, experts)", "bound": "hbm",
            "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": ach / peaks["hbm_gbs"],
            "traffic": None, "peak_note": peak_note}


def kernels_per_call(s):
    """Kernels one moe_layer_fwd launches (the library's own, no memsets or copies)."""
    tc_router = s.x_dtype == "bf16" and s.T >= 128 and s.E in (16, 32, 48, 64, 80)
    router = 2 if tc_router else 1                     # weight split + router, or SIMT router
    if s.w_format == "int4":
        if s.T * s.k <= 8 and s.x_dtype == "bf16" and s.d % 256 == 0 and s.f % 256 == 0:
            return 1  # the single-launch serving kernel (with the expert cache's plan and fill)
        if s.T * s.k <= 64:
            # no permutation: shared gate/up and down (second stream), int4 gate/up, int4
            # down with the combine (or, off the tensor-core shapes, the shared down with
            # the combine; the combine kernel without a shared expert)
            return router + 2 + (2 if s.F else 1)
        # permute, shared gate/up, int4 gate/up, int4 down, shared down + combine
        return router + 1 + (4 if s.F else 2) + (0 if s.F else 1)
    # permute, then either the shared gate/up (second stream) and one launch with the
    # routed gate/up, shared down and the chained routed down, or a gate/up launch and a
    # down launch; combine
    return router + 1 + 2 + 1


# Kernels one moe_layer_bwd launches: padded layout with the row gather, five grouped GEMMs
# (dgrad down; gate/up recompute with the SwiGLU backward; dgrad gate/up; two weight
# gradients), router backward + dx, router weight gradient.
KERNELS_PER_BWD = 8


def train_algorithmic(s):
    """FLOPs and bytes of one training step of the layer: the forward's, plus the
    backward's input and weight gradients (twice the expert GEMM FLOPs, and the
    router's two products over the winners); bytes add the weights read again, the
    fp32 weight gradients written, dout and x read, dx written."""
    f_fwd, b_fwd = layer_algorithmic(s)
    expert_flops = 2 * 3 * s.d * s.f * s.T * s.k + 2 * 3 * s.d * s.F * s.T
    f_bwd = 2 * expert_flops + 2 * 2 * s.T * s.k * s.d
    hit = min(s.E, s.T * s.k)
    w_bytes = hit * 3 * s.d * s.f * 2 + 3 * s.d * s.F * 2 + s.E * s.d * 4
    g_bytes = (hit * 3 * s.d * s.f + 3 * s.d * s.F + s.E * s.d) * 4
    b_bwd = w_bytes + g_bytes + 3 * s.T * s.d * 2
    return f_fwd + f_bwd, b_fwd + b_bwd


def bwd_stage_work(s, stage):
    """(FLOPs, HBM bytes that must move) of one backward GEMM stage, algorithmic:
    its weights or fp32 weight gradients, and its activation operands and outputs
    once (padding rows not counted)."""
    P, T, d, f, F = s.T * s.k, s.T, s.d, s.f, s.F
    hit = min(s.E, P)
    wd, wgu = hit * d * f + d * F, hit * 2 * f * d + 2 * F * d   # weight elements
    table = {
        # dh = dout Wd (P + T rows of dout in, dh out)
        "bwd_dgrad_down": (2 * P * d * f + 2 * T * d * F, wd * 2 + (P + T) * d * 2 + (P * f + T * F) * 2),
        # pre-activations recomputed, SwiGLU backward: x rows and dh in; (da, db) and g h out
        "bwd_recompute_swiglu": (2 * P * d * 2 * f + 2 * T * d * 2 * F,
                                 wgu * 2 + (P + T) * d * 2 + (P * f + T * F) * 2 * 2 + (P * 2 * f + T * 2 * F) * 2),
        # dx rows = (da, db) Wgu
        "bwd_dgrad_gate_up": (2 * P * 2 * f * d + 2 * T * 2 * F * d,
                              wgu * 2 + (P * 2 * f + T * 2 * F) * 2 + (P + T) * d * 2),
        # dWd = dout^T (g h): fp32 gradients out
        "bwd_wgrad_down": (2 * P * d * f + 2 * T * d * F, wd * 4 + (P + T) * d * 2 + (P * f + T * F) * 2),
        # dWgu = (da, db)^T x: fp32 gradients out
        "bwd_wgrad_gate_up": (2 * P * 2 * f * d + 2 * T * 2 * F * d,
                              wgu * 4 + (P * 2 * f + T * 2 * F) * 2 + (P + T) * d * 2),
    }
    return table.get(stage)


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=sorted(WORKLOADS) + ["attn"], default="nano")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-sample-worker", default=None, help=argparse.SUPPRESS)
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target CPU time of the oracle baseline sample (0: none)")
    return p.parse_args()


# ----------------------------------------------------------------------------- helpers

# name -> (case used for the seeds, shape, workload label, metric)
WORKLOADS = {
    "nano": ("nano", CONFIGS["nano"], "nano_moe_layer_fwd_T8192", METRIC),
    "skew": ("skew", CONFIGS["skew"], "skewed_zipf1.2_moe_layer_fwd_T8192_50_steps",
             "Skewed-load MoE-layer fwd + bias update tokens/s (Zipf 1.2 router offsets), % roofline"),
    "stack": ("stack", CONFIGS["stack"], "stack_23_moe_layers_T8192",
              "23-layer MoE stack fwd tokens/s per stack forward, % roofline"),
    "tiny": ("tiny", CONFIGS["tiny"], "tiny_moe_layer_fwd_T64", "tiny MoE-layer fwd tokens/s"),
    "train": ("nano", CONFIGS["nano"], "nano_moe_layer_fwd_bwd_T8192",
              "MoE-layer training step (fwd + bias update + bwd) tokens/s (T=8192,d=1024,64x512 top-2+2048 "
              "shared), % roofline"),
    "decode1": ("decode", CONFIGS["decode"].replace(T=1), "top1_int4_decode_T1",
                "Top-1 int4 serving decode tokens/s (T=1), % HBM roofline"),
    "decode8": ("decode", CONFIGS["decode"].replace(T=8), "top1_int4_decode_T8",
                "Top-1 int4 serving decode tokens/s (T=8), % HBM roofline"),
    "decode64": ("decode", CONFIGS["decode"].replace(T=64), "top1_int4_decode_T64",
                 "Top-1 int4 serving decode tokens/s (T=64), % HBM roofline"),
    "cache8": ("decode", CONFIGS["decode"].replace(T=8, skew_zipf_s=1.2),
               "top1_int4_decode_T8_expert_cache_16_of_64_zipf1.2",
               "Top-1 int4 serving tokens/s through the GPU expert cache (T=8, 16 of 64 experts in HBM, "
               "Zipf 1.2 routing), hit rate"),
    "cache8u": ("decode", CONFIGS["decode"].replace(T=8),
                "top1_int4_decode_T8_expert_cache_16_of_64_uniform",
                "Top-1 int4 serving tokens/s through the GPU expert cache (T=8, 16 of 64 experts in HBM, "
                "unskewed routing), hit rate"),
    "cache1": ("decode", CONFIGS["decode"].replace(T=1, skew_zipf_s=1.2),
               "top1_int4_decode_T1_expert_cache_4_of_64_zipf1.2",
               "Top-1 int4 serving tokens/s through the GPU expert cache (T=1, 4 of 64 experts in HBM, "
               "Zipf 1.2 routing), hit rate"),
}
CACHE_SLOTS = {"cache8": 16, "cache8u": 16, "cache1": 4}
CACHE_BATCHES = 64  # distinct resident token batches the timed steps cycle through


ATTN_METRIC = ("Attention block fwd tokens/s (4x GQA, per-head QK-norm, batch 4 x seq 2048, d=1024, "
               "8 query / 2 key-value heads of 128), % roofline")


def workload_shape(name):
    return WORKLOADS[name][1]


def attn_algorithmic(s):
    """FLOPs and bytes of one attention block forward: the projections, the causal
    attention (scores and the weighted values over the causal triangle of each
    sequence), weights and the tokens in and out."""
    hd, C, HO = s.head_dim, (s.n_head + 2 * s.n_kv_head) * s.head_dim, s.n_head * s.head_dim
    proj = 2 * s.T * s.d * C + 2 * s.T * HO * s.d
    attn = s.batch * s.n_head * 4 * hd * (s.seq * (s.seq + 1) // 2)
    nbytes = 2 * (C * s.d + s.d * HO) + 2 * 2 * s.T * s.d
    return proj, attn, nbytes


def config_block(name, n):
    s = workload_shape(name)
    cfg = {"workload": WORKLOADS[name][2],
           "T": s.T, "d": s.d, "E": s.E, "f": s.f, "F": s.F, "k": s.k, "renorm": bool(s.renorm),
           "routed_weights": s.w_format,
           "bias_update": s.w_format != "int4", "tokens": "batch 4 x seq 2048" if s.T == 8192 else f"{s.T}",
           "layers": s.layers, "l2": "512 MiB write before every timed step (L2 129 MB)",
           "parallelism": f"dp{n} replicas, per-expert load all-reduce" if n > 1 else "dp1"}
    return cfg


def layer_algorithmic(s, loads_hit=None):
    """FLOPs and bytes one layer forward must move (weights of the experts hit, shared
    and router weights, x in, out)."""
    flops = 2 * s.T * s.d * s.E + 2 * 3 * s.d * s.f * s.T * s.k + 2 * 3 * s.d * s.F * s.T
    hit = min(s.E, s.T * s.k) if loads_hit is None else int(loads_hit)
    if s.w_format == "int4":
        expert = 3 * s.d * s.f // 2 + 3 * s.d * s.f // 32 * 2
    else:
        expert = 3 * s.d * s.f * 2
    nbytes = hit * expert + 3 * s.d * s.F * 2 + s.E * s.d * 4 + 2 * s.T * s.d * 2
    return flops, nbytes


def load_peaks():
    try:
        with open(PEAKS_FILE) as fh:
            pk = json.load(fh)
        return pk, "of measured"
    except (OSError, ValueError):
        return FALLBACK_PEAKS, "of fallback"


def gemm_source_hash():
    h = hashlib.sha256()
    for f in ("gemm.cu", "ptx.cuh"):
        with open(os.path.join(ROOT, "aux_loss_free_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def read_traffic(path=TRAFFIC_FILE):
    """DRAM bytes per launch of the dominant GEMM from the committed ncu summary, if it
    was taken on the current kernel source (else None)."""
    try:
        kv = {}
        with open(path) as fh:
            for line in fh:
                if ":" in line:
                    a, b = line.split(":", 1)
                    kv[a.strip()] = b.strip()
        if kv.get("kernel_source_sha256_16") != gemm_source_hash():
            return None
        return float(kv["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 20 ms in the background."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.rows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-i", str(index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.rows.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        inside = [p for (t, p) in self.rows if t0 <= t <= t1] or [p for (_, p) in self.rows]

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        mx = [num(p[2]) for p in inside if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside),
                "power_w_max": max((num(p[3]) or 0.0) for p in inside)}


# ----------------------------------------------------------------------------- oracle arm

def oracle_sample_runner(name, seed):
    """Returns run(ntok) -> seconds for the oracle's layer forward on the first ntok
    tokens of the workload (fp64 oracle, as it stands)."""
    from oracle import moe_oracle as O

    s = workload_shape(name)
    host = make_layer(s, WORKLOADS[name][0], seed)
    bf = lambda b: f32_from_bf16_bits(b).astype(np.float64)  # noqa: E731
    W = {k: bf(host[k]) for k in ("w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down")}
    if s.w_format == "int4":
        # The serving model's routed experts are the int4 round trip of the bf16 ones
        # (quantised once, outside the timed calls).
        for key in ("w_gate", "w_up", "w_down"):
            G, R, K = W[key].shape
            packed, scale, _ = O.quantize_int4_g32(W[key].reshape(-1, K).astype(np.float32))
            W[key] = O.dequantize_int4_g32(packed, scale).reshape(G, R, K)
    x = host["x"]
    xv = bf(x) if x.dtype == np.uint16 else x.astype(np.float64)

    dout = bf(make_output_grad(s, WORKLOADS[name][0], seed)) if name == "train" else None

    def run(ntok):
        t0 = time.perf_counter()
        O.layer_forward(xv[:ntok], host["w_router"], host["bias"], W["w_gate"], W["w_up"],
                        W["w_down"], W["s_gate"], W["s_up"], W["s_down"], k=s.k, renorm=s.renorm,
                        logit_offset=host["logit_offset"], gamma=host["gamma"],
                        x_is_bf16=x.dtype == np.uint16)
        if dout is not None:
            O.layer_backward(xv[:ntok], host["w_router"], host["bias"], W["w_gate"], W["w_up"],
                             W["w_down"], W["s_gate"], W["s_up"], W["s_down"], dout[:ntok], s.k,
                             renorm=s.renorm, logit_offset=host["logit_offset"])
        return time.perf_counter() - t0
    return run


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def timed_oracle_sample(name, seed, seconds):
    """(tokens done, seconds spent, tokens per call) of the oracle on the workload."""
    run = oracle_sample_runner(name, seed)
    s = workload_shape(name)
    ntok = min(s.T, 128 if name == "train" else 1024)
    run(min(ntok, 64))  # warm the BLAS threads
    done, spent = 0, 0.0
    while spent < seconds and done < 64 * s.T:
        spent += run(ntok)
        done += ntok
    return done, spent, ntok


def one_thread_baseline(name, seed, seconds):
    """The same oracle sample on one host thread: a child process (a fresh interpreter,
    nothing forked from a process that holds a CUDA context) with every BLAS thread
    pool set to one thread before numpy loads."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1", VECLIB_MAXIMUM_THREADS="1")
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-sample-worker", name, "--seed", str(seed),
           "--cpu-seconds", str(seconds)]
    try:
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=seconds * 6 + 120)
        done, spent, ntok = json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as exc:  # the main measurement stands without it
        return {"error": f"one-thread sample failed: {exc!r}"[:200]}
    s = workload_shape(name)
    return {"value": done / spent * (1.0 / max(1, s.layers)), "unit": "tokens/s", "cores": 1,
            "sample": f"{done} tokens in calls of {ntok}, BLAS on one thread, {spent:.1f} s"}


def cpu_baseline(name, seed, seconds):
    if seconds <= 0:  # --cpu-seconds 0: no oracle timing (profiling runs)
        return None
    run = oracle_sample_runner(name, seed)
    s = workload_shape(name)
    ntok = min(s.T, 128 if name == "train" else 1024)
    run(min(ntok, 64))  # warm the BLAS threads
    done, spent = 0, 0.0
    while spent < seconds and done < 64 * s.T:
        spent += run(ntok)
        done += ntok
    return {"value": done / spent * (1.0 / max(1, s.layers)), "unit": "tokens/s", "cores": cpu_cores(),
            "kind": "oracle",
            "sample": f"{done} tokens as {done // ntok} oracle layer "
                      f"{'forward+backward passes' if name == 'train' else 'forwards'} of {ntok} tokens of the "
                      f"{name} workload (fp64 numpy, BLAS on all {cpu_cores()} visible cores), "
                      f"{spent:.1f} s" + (f"; per stack forward of {s.layers} layers" if s.layers > 1 else ""),
            "one_thread": one_thread_baseline(name, seed, max(2.0, min(8.0, seconds / 2)))}


def reference_arm(args, rank, world):
    if rank != 0:
        return
    run = oracle_sample_runner(args.workload, args.seed)
    s = workload_shape(args.workload)
    cal = min(s.T, 256)
    t_cal = run(cal)
    budget = 150.0 / max(1, args.steps + args.warmup)
    ntok = int(min(s.T, max(1, cal * budget / max(t_cal, 1e-6))))
    if ntok >= 32:
        ntok = ntok // 32 * 32
    for _ in range(args.warmup):
        run(ntok)
    times = [run(ntok) for _ in range(args.steps)]
    total = sum(times)
    value = ntok * args.steps / total / max(1, s.layers)
    line = {"impl": "reference", "metric": WORKLOADS[args.workload][3], "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_block(args.workload, world),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "kind": "oracle", "cores": cpu_cores(),
                             "sample": f"each step: oracle layer "
                                       f"{'forward+backward' if args.workload == 'train' else 'forward'}"
                                       f" of {ntok} of the {s.T} tokens"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU arm

def gpu_arm(args, rank, world, dist):
    import torch

    import aux_loss_free_gb300 as M
    from aux_loss_free_gb300.dp import dp_bias_update
    from aux_loss_free_gb300.layer import LayerOnDevice, to_device_tokens

    M.load_library()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    s = workload_shape(args.workload)
    name = args.workload
    case = WORKLOADS[name][0]
    nlayers = s.layers
    update = s.w_format != "int4"   # serving does not move the bias
    layers = [LayerOnDevice(s, make_layer(s, case, args.seed, layer=l, with_tokens=False), dev)
              for l in range(nlayers)]
    bias0 = [L.bias.clone() for L in layers]
    host_x = make_tokens(s, case, args.seed + rank)
    x0 = to_device_tokens(host_x, dev)
    mids = [torch.empty(s.T, s.d, dtype=torch.bfloat16, device=dev) for _ in range(max(0, nlayers - 1))]
    out0 = torch.empty(s.T, s.d, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    load = torch.empty(s.E, dtype=torch.int32, device=dev)
    dbg_load = M.make_debug(load=load)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step(x_in, out):
        """One pass of the whole path: every layer's forward and bias update."""
        cur = x_in
        for l, L in enumerate(layers):
            nxt = out if l == nlayers - 1 else mids[l]
            res = cur if nlayers > 1 else None
            if world > 1 and update:
                # Data-parallel replicas: local loads, global sum, identical update.
                L.forward(cur, nxt, update_bias=False, residual=res, debug=dbg_load)
                dp_bias_update(load, L.bias, L.gamma)
            else:
                L.forward(cur, nxt, update_bias=update, residual=res)
            cur = nxt
        return out

    for _ in range(args.warmup):
        step(x0, out0)
    torch.cuda.synchronize(dev)
    if M.moe_device_status() != 0:
        raise RuntimeError("device status set during warm-up")

    # ---------------------------------------------------------------- timed region
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    time.sleep(0.1)
    K = args.steps
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    # Stage events on every 10th layer call only: each event costs ~2 us of stream time.
    M.moe_profile_start(K * nlayers // PROFILE_PERIOD + 1, PROFILE_PERIOD)
    t_wall0 = time.time()
    for i in range(K):
        flush.zero_()
        ev0[i].record(stream)
        step(x0, out0)
        ev1[i].record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    if dist:
        dist.barrier()
    stages_ms, calls = M.moe_profile_stop()
    time.sleep(0.05)
    sampler.stop()
    step_ms = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
    total_ms = sum(step_ms)
    if dist:
        t = torch.tensor([total_ms], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    status = M.moe_device_status()

    # ---------------------------------------------------------------- end to end
    # The same steps through the public call with host buffers: every step copies its
    # tokens in from pinned host memory and reads its output back, both inside the
    # timed region.  Copies run on a second stream, double-buffered, overlapping the
    # neighbouring steps' compute as an input pipeline would.
    Ke = max(3, min(K, 100))
    hx = [torch.empty(s.T, s.d, dtype=x0.dtype, pin_memory=True) for _ in range(2)]
    for b in hx:
        b.copy_(x0.cpu())
    hout = [torch.empty(s.T, s.d, dtype=torch.bfloat16, pin_memory=True) for _ in range(2)]
    din = [torch.empty_like(x0) for _ in range(2)]
    dout = [torch.empty(s.T, s.d, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    cs = torch.cuda.Stream(dev)      # host -> device copies
    ds = torch.cuda.Stream(dev)      # device -> host copies (a second copy engine)
    h2d = [torch.cuda.Event() for _ in range(Ke)]
    done = [torch.cuda.Event() for _ in range(Ke)]
    d2h = [torch.cuda.Event() for _ in range(Ke)]
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e_start.record(cs)
    for i in range(Ke):
        b = i % 2
        with torch.cuda.stream(cs):
            if i >= 2:
                cs.wait_event(done[i - 2])   # din[b] free again
            din[b].copy_(hx[b], non_blocking=True)
            h2d[i].record(cs)
        stream.wait_event(h2d[i])
        if i >= 2:
            stream.wait_event(d2h[i - 2])    # dout[b] read back already
        # No L2 flush here: every step copies fresh tokens in and the layer's weights
        # (214 MB for the Nano layer) exceed the 129 MB L2 by themselves.
        step(din[b], dout[b])
        done[i].record(stream)
        with torch.cuda.stream(ds):
            ds.wait_event(done[i])
            hout[b].copy_(dout[b], non_blocking=True)
            d2h[i].record(ds)
    cs.wait_event(d2h[Ke - 1])
    e_end.record(cs)
    torch.cuda.synchronize(dev)
    e2e_ms = e_start.elapsed_time(e_end) / Ke

    # Load trajectory (skewed workload: the configured 50 steps from the initial bias)
    # and the number of experts hit, read after the timed region.
    for L, b in zip(layers, bias0):
        L.bias.copy_(b)
    nsteps = max(1, s.steps)
    loads = torch.empty(nsteps, s.E, dtype=torch.int32, device=dev)
    for i in range(nsteps):
        L0 = layers[0]
        L0.forward(x0, out0 if nlayers == 1 else mids[0], update_bias=update,
                   residual=x0 if nlayers > 1 else None, debug=M.make_debug(load=loads[i]))
    ld = loads.cpu().numpy().astype(np.float64)
    hit = int((ld[0] > 0).sum())
    traj = (ld.max(axis=1) / ld.mean(axis=1)).tolist()
    dead = (ld == 0).mean(axis=1).tolist()  # fraction of experts with no pair, per step

    if rank != 0:
        return
    peaks, peak_note = load_peaks()
    flops, nbytes = layer_algorithmic(s, hit)
    tokens_per_s = world * s.T * K / (total_ms / 1e3)
    ms_step = total_ms / K
    roof_s = nlayers * max(flops / (peaks["bf16_tflops"] * 1e12), nbytes / (peaks["hbm_gbs"] * 1e9))
    # Dominant kernel: the longest stage.  When the layer forks the routing onto a
    # second stream that is the chained launch (routed gate/up beside the shared down
    # projection, the routed down projection chained behind); the shared-expert gate/up
    # launch that runs beside the routing is reported next to it.  Otherwise the
    # combined gate/up launch.
    routed_gu = 2 * s.T * s.k * s.d * 2 * s.f
    routed_dn = 2 * s.T * s.k * s.f * s.d
    shared_gu = 2 * s.T * s.d * 2 * s.F
    shared_dn = 2 * s.T * s.F * s.d
    extra_rooflines = {}
    if "routed_ffn_shared_down" in stages_ms:
        dom_name = ("grouped_gemm_kernel (chained launch: routed gate/up + shared down projection, "
                    "routed down projection chained)")
        gu_flops = routed_gu + shared_dn + routed_dn
        gu_ms = stages_ms["routed_ffn_shared_down"] / max(1, calls)
        sg_ms = stages_ms["shared_gate_up"] / max(1, calls)
        sg_ach = shared_gu / (sg_ms / 1e3) / 1e12
        extra_rooflines["shared_gate_up"] = {
            "kernel": "grouped_gemm_kernel (shared-expert gate/up launch, concurrent with routing)",
            "bound": "tensor", "achieved": sg_ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": sg_ach / peaks["bf16_tflops"], "traffic": read_traffic(SHARED_TRAFFIC_FILE),
            "flops_per_launch": shared_gu, "avg_launch_us": sg_ms * 1e3}
    else:
        dom_name = "grouped_gemm_kernel (gate/up launch: routed groups + shared)"
        gu_flops = routed_gu + shared_gu
        gu_ms = stages_ms.get("gemm_gate_up", float("nan")) / max(1, calls)
    achieved = gu_flops / (gu_ms / 1e3) / 1e12
    traffic = read_traffic() if "routed_ffn_shared_down" in stages_ms else None
    clocks = sampler.summary(t_wall0, t_wall1)
    line = {
        "metric": WORKLOADS[name][3], "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_block(name, world),
        "layer_roofline": {"flops_per_layer": flops, "bytes_per_layer": nbytes,
                           "roofline_us": roof_s * 1e6, "measured_us": ms_step * 1e3,
                           "frac": roof_s / (ms_step / 1e3), "peak": peak_note,
                           "frac_sustained": nlayers * max(
                               flops / (peaks["bf16_tflops_sustained"] * 1e12),
                               nbytes / (peaks["hbm_gbs"] * 1e9)) / (ms_step / 1e3),
                           "bound": "tensor" if flops / (peaks["bf16_tflops"] * 1e12) >
                           nbytes / (peaks["hbm_gbs"] * 1e9) else "hbm"},
        "roofline": {"kernel": dom_name,
                     "bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                     "traffic": traffic, "peak_note": peak_note + " (burst)",
                     "frac_sustained": achieved / peaks["bf16_tflops_sustained"],
                     "flops_per_launch": gu_flops, "avg_launch_us": gu_ms * 1e3},
        "stages_us": {k: v * 1e3 / max(1, calls) for k, v in stages_ms.items()},
        "other_rooflines": extra_rooflines,
        "step_us": {"median": statistics.median(step_ms) * 1e3, "min": min(step_ms) * 1e3,
                    "max": max(step_ms) * 1e3, "note": "per timed step (CUDA events); ms_per_step is the mean"},
        "e2e": {"value": world * s.T / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": int(hx[0].numel() * hx[0].element_size()),
                "d2h_bytes_per_step": int(hout[0].numel() * hout[0].element_size()),
                "copies": "pinned host buffers; H2D and D2H on their own streams overlapped with compute (double-buffered); no L2 flush (weights exceed L2)"},
        "gpu_launches": K * nlayers * kernels_per_call(s),
        "clocks": clocks,
        "device_status": status,
        "experts_hit": hit,
    }
    if s.steps > 1:
        line["load_max_over_mean"] = {"first": traj[0], "last": traj[-1],
                                      "per_step": [round(v, 3) for v in traj]}
        line["dead_expert_fraction"] = {"first": dead[0], "last": dead[-1],
                                        "per_step": [round(v, 4) for v in dead]}
    if s.w_format == "int4":
        # Serving is bound by weight bytes: report the HBM roofline of the layer.
        line["roofline"] = {"kernel": "whole top-1 serving layer", "bound": "hbm",
                            "achieved": nbytes / (ms_step / 1e3) / 1e9, "peak": peaks["hbm_gbs"],
                            "unit": "GB/s", "frac": nbytes / (ms_step / 1e3) / 1e9 / peaks["hbm_gbs"],
                            "traffic": None, "peak_note": peak_note, "bytes_per_step": nbytes}
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(name if nlayers == 1 else "nano", args.seed,
                                            args.cpu_seconds)
    print(json.dumps(line), flush=True)


def gpu_train_arm(args, rank, world, dist):
    """Training step of the Nano layer: forward (routing state saved) with the bias
    update, then the backward for a seeded output gradient."""
    import torch

    import aux_loss_free_gb300 as M
    from aux_loss_free_gb300.dp import dp_bias_update
    from aux_loss_free_gb300.layer import (LayerGrads, LayerOnDevice, SavedForward, attach_backward,
                                           layer_backward, to_device_bf16, to_device_tokens)

    M.load_library()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    name = args.workload
    s = workload_shape(name)
    case = WORKLOADS[name][0]
    layer = attach_backward(LayerOnDevice(s, make_layer(s, case, args.seed, with_tokens=False), dev))
    x0 = to_device_tokens(make_tokens(s, case, args.seed + rank), dev)
    g0 = to_device_bf16(make_output_grad(s, case, args.seed + rank), dev)
    saved = SavedForward(s.T, s.E, s.k, dev)
    grads = LayerGrads(layer)
    out0 = torch.empty(s.T, s.d, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step(x_in, dout, out):
        if world > 1:
            layer.forward(x_in, out, update_bias=False, debug=saved.debug)
            dp_bias_update(saved.load, layer.bias, layer.gamma)
        else:
            layer.forward(x_in, out, update_bias=True, debug=saved.debug)
        layer_backward(layer, x_in, saved, dout, grads)

    for _ in range(args.warmup):
        step(x0, g0, out0)
    torch.cuda.synchronize(dev)
    if M.moe_device_status() != 0:
        raise RuntimeError("device status set during warm-up")

    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    time.sleep(0.1)
    K = args.steps
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    # An odd sampling period alternates the recorded calls between forward and backward
    # (every call of a short run).
    period = PROFILE_PERIOD + 1 if 2 * K >= 4 * (PROFILE_PERIOD + 1) else 1
    M.moe_profile_start(2 * K // period + 2, period)
    t_wall0 = time.time()
    for i in range(K):
        flush.zero_()
        ev0[i].record(stream)
        step(x0, g0, out0)
        ev1[i].record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    if dist:
        dist.barrier()
    stages_ms, stage_calls = M.moe_profile_stop(per_stage_calls=True)
    time.sleep(0.05)
    sampler.stop()
    step_ms = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
    total_ms = sum(step_ms)
    if dist:
        t = torch.tensor([total_ms], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    status = M.moe_device_status()

    # End to end: x and dout in from pinned host memory, dx back, every step inside
    # the timed region (the weight gradients stay on the device for the optimizer).
    Ke = max(3, min(K, 50))
    hx = torch.empty(s.T, s.d, dtype=x0.dtype, pin_memory=True)
    hx.copy_(x0.cpu())
    hg = torch.empty(s.T, s.d, dtype=torch.bfloat16, pin_memory=True)
    hg.copy_(g0.cpu())
    hdx = torch.empty(s.T, s.d, dtype=torch.bfloat16, pin_memory=True)
    dx_, dg_ = torch.empty_like(x0), torch.empty_like(g0)
    torch.cuda.synchronize(dev)
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    for _ in range(Ke):
        dx_.copy_(hx, non_blocking=True)
        dg_.copy_(hg, non_blocking=True)
        step(dx_, dg_, out0)
        hdx.copy_(grads.dx, non_blocking=True)
    e_end.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e_start.elapsed_time(e_end) / Ke

    if rank != 0:
        return
    peaks, peak_note = load_peaks()
    flops, nbytes = train_algorithmic(s)
    ms_step = total_ms / K
    roof_s = max(flops / (peaks["bf16_tflops"] * 1e12), nbytes / (peaks["hbm_gbs"] * 1e9))
    per_call = {k: v / max(1, stage_calls.get(k, 1)) for k, v in stages_ms.items()}
    # Dominant kernel: the slowest backward GEMM stage, against the bound its
    # algorithmic FLOPs and bytes set.
    cands = [(per_call[k], k) for k in per_call if bwd_stage_work(s, k)]
    if not cands:
        raise RuntimeError("no backward stage was recorded")
    dom_ms, dom = max(cands)
    fl, by = bwd_stage_work(s, dom)
    t_fl = fl / (peaks["bf16_tflops"] * 1e12)
    t_by = by / (peaks["hbm_gbs"] * 1e9)
    if t_fl >= t_by:
        roof = {"bound": "tensor", "achieved": fl / (dom_ms / 1e3) / 1e12, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": by / (dom_ms / 1e3) / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof.update({"kernel": f"grouped_gemm_kernel ({dom} launch)", "frac": roof["achieved"] / roof["peak"],
                 "traffic": read_traffic(TRAIN_TRAFFIC_FILE) if dom == "bwd_wgrad_gate_up" else None, "peak_note": peak_note + (" (burst)" if roof["unit"] == "TFLOP/s" else ""),
                 "flops_per_launch": fl, "bytes_per_launch": by, "avg_launch_us": dom_ms * 1e3})
    fwd_k = kernels_per_call(s)
    line = {
        "metric": WORKLOADS[name][3], "value": world * s.T * K / (total_ms / 1e3), "unit": "tokens/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(config_block(name, world), step="fwd + bias update + bwd (dx, fp32 weight grads)"),
        "layer_roofline": {"flops_per_step": flops, "bytes_per_step": nbytes, "roofline_us": roof_s * 1e6,
                           "measured_us": ms_step * 1e3, "frac": roof_s / (ms_step / 1e3), "peak": peak_note,
                           "frac_sustained": max(flops / (peaks["bf16_tflops_sustained"] * 1e12),
                                                 nbytes / (peaks["hbm_gbs"] * 1e9)) / (ms_step / 1e3),
                           "bound": "tensor" if flops / (peaks["bf16_tflops"] * 1e12) >
                           nbytes / (peaks["hbm_gbs"] * 1e9) else "hbm"},
        "roofline": roof,
        "stages_us": {k: v * 1e3 for k, v in per_call.items()},
        "e2e": {"value": world * s.T / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": int(2 * hx.numel() * hx.element_size()),
                "d2h_bytes_per_step": int(hdx.numel() * hdx.element_size()),
                "copies": "x and dout from pinned host memory, dx back, on the compute stream; weight "
                          "gradients stay on the device"},
        "gpu_launches": K * (fwd_k + KERNELS_PER_BWD),
        "clocks": sampler.summary(t_wall0, t_wall1),
        "device_status": status,
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(name, args.seed, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def gpu_cache_arm(args, rank, world, dist):
    """Top-1 int4 serving through the GPU expert cache: every step routes a different
    batch of tokens (cycling through CACHE_BATCHES resident batches), so the cache sees
    a stream of routing results; the all-resident layer is timed on the same batches."""
    import torch

    import aux_loss_free_gb300 as M
    from aux_loss_free_gb300.layer import ExpertCache, LayerOnDevice, to_device_tokens

    M.load_library()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    name = args.workload
    s = workload_shape(name)
    case = WORKLOADS[name][0]
    slots = CACHE_SLOTS[name]
    layer = LayerOnDevice(s, make_layer(s, case, args.seed, with_tokens=False), dev)
    cache = ExpertCache(layer, slots)
    batches = [to_device_tokens(make_tokens(s, case, args.seed + 1000 * rank + b), dev) for b in range(CACHE_BATCHES)]
    out0 = torch.empty(s.T, s.d, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    expert_bytes = sum(int(t.numel() * t.element_size()) // s.E for t in cache.host.values())

    def run(fn, K, warm, profile=False):
        for i in range(warm):
            fn(batches[i % CACHE_BATCHES], out0)
        torch.cuda.synchronize(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        if profile:
            M.moe_profile_start(K + 1, 1)
        t0 = time.time()
        for i in range(K):
            flush.zero_()
            ev[i][0].record(stream)
            fn(batches[(warm + i) % CACHE_BATCHES], out0)
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        t1 = time.time()
        stages = M.moe_profile_stop(per_stage_calls=True) if profile else None
        return sum(a.elapsed_time(b) for a, b in ev), stages, t0, t1

    K = args.steps
    run(lambda x, o: layer.forward(x, o, update_bias=False), 0, args.warmup)
    res_ms, _, _, _ = run(lambda x, o: layer.forward(x, o, update_bias=False), K, 0)
    cache.reset()
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    time.sleep(0.1)
    for i in range(args.warmup):
        cache.forward(batches[i % CACHE_BATCHES], out0)
    st0, _, _, _ = cache.read()
    if dist:
        dist.barrier()
    total_ms, _, tw0, tw1 = run(lambda x, o: cache.forward(x, o), K, 0)
    st1, _, _, _ = cache.read()
    sampler.stop()
    # Stage times from a separate pass (each stage event adds ~2 us to the stream).
    _, (stages_ms, stage_calls), _, _ = run(lambda x, o: cache.forward(x, o), min(K, 50), 0, profile=True)
    if dist:
        t = torch.tensor([total_ms], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    status = M.moe_device_status()
    # Host -> device bandwidth of a plain pinned copy: the fill path's ceiling.
    hsrc = torch.empty(256 << 20, dtype=torch.uint8, pin_memory=True)
    ddst = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    ddst.copy_(hsrc, non_blocking=True)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(4):
        ddst.copy_(hsrc, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    link_gbs = 4 * hsrc.numel() / (e0.elapsed_time(e1) / 1e3) / 1e9
    # End to end: tokens in from pinned memory, output back, each step.
    Ke = max(3, min(K, 100))
    hxs = []
    for b in batches:  # every step's tokens come from host memory, as served
        h = torch.empty(s.T, s.d, dtype=b.dtype, pin_memory=True)
        h.copy_(b.cpu())
        hxs.append(h)
    hx = hxs[0]
    hout = torch.empty(s.T, s.d, dtype=torch.bfloat16, pin_memory=True)
    din = torch.empty_like(batches[0])
    torch.cuda.synchronize(dev)
    ee0, ee1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ee0.record(stream)
    for i in range(Ke):
        din.copy_(hxs[i % CACHE_BATCHES], non_blocking=True)
        cache.forward(din, out0)
        hout.copy_(out0, non_blocking=True)
    ee1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = ee0.elapsed_time(ee1) / Ke
    if rank != 0:
        return
    peaks, peak_note = load_peaks()
    hits, misses = st1["hits"] - st0["hits"], st1["misses"] - st0["misses"]
    fill_bytes = st1["bytes"] - st0["bytes"]
    ms_step = total_ms / K
    fetch_ms = stages_ms.get("cache_fetch", float("nan")) / max(1, stage_calls.get("cache_fetch", 1))
    fill_gbs = (fill_bytes / K) / (fetch_ms / 1e3) / 1e9 if fetch_ms == fetch_ms and fetch_ms > 0 else None
    fused = "serve_fused" in stages_ms  # the plan and the fill run inside the one serving launch
    # Weight bytes a step must read: the distinct experts it uses (from HBM slots) and
    # the shared expert, as in the serving workloads' HBM roofline.
    used_per_step = (hits + misses) / K
    flops, _ = layer_algorithmic(s)
    nbytes = int(used_per_step * (3 * s.d * s.f // 2 + 3 * s.d * s.f // 32 * 2) + 3 * s.d * s.F * 2
                 + s.E * s.d * 4 + 4 * s.T * s.d)
    line = {
        "metric": WORKLOADS[name][3], "value": world * s.T * K / (total_ms / 1e3), "unit": "tokens/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int4 weights, bf16 activations", "data": "synthetic",
        "config": dict(config_block(name, world), slots=slots, token_batches=CACHE_BATCHES,
                       weights="int4 experts in pinned host memory, slots in HBM"),
        "cache": {"hit_rate": hits / max(1, hits + misses), "hits": hits, "misses": misses,
                  "evictions": st1["evictions"] - st0["evictions"], "bytes_per_step": fill_bytes / K,
                  "expert_bytes": expert_bytes, "fetch_us_per_step": fetch_ms * 1e3,
                  "resident_us_per_step": res_ms / K * 1e3,
                  "overflow": st1["overflow"] - st0["overflow"]},
        "roofline": ({"kernel": "cache fill (plan + copy kernels, host memory -> HBM slots)", "bound": "link",
                      "achieved": fill_gbs, "peak": link_gbs, "unit": "GB/s",
                      "frac": (fill_gbs / link_gbs) if fill_gbs else None, "traffic": None,
                      "peak_note": "of a pinned host-to-device copy measured in this run"} if not fused else
                     serve_step_roofline(fill_bytes / K, nbytes, ms_step, link_gbs, peaks, peak_note)),
        "layer_roofline": {"bytes_per_step": nbytes, "roofline_us": nbytes / (peaks["hbm_gbs"] * 1e9) * 1e6,
                           "measured_us": ms_step * 1e3,
                           "frac": nbytes / (peaks["hbm_gbs"] * 1e9) / (ms_step / 1e3), "peak": peak_note,
                           "bound": "hbm"},
        "stages_us": {k: v * 1e3 / max(1, stage_calls.get(k, 1)) for k, v in stages_ms.items()},
        "e2e": {"value": world * s.T / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": int(hx.numel() * hx.element_size()),
                "d2h_bytes_per_step": int(hout.numel() * hout.element_size()),
                "copies": "tokens in from pinned memory and the output back on the compute stream"},
        # the cache's plan and copy kernels, unless they ran inside the single serving launch
        "gpu_launches": K * (kernels_per_call(s) + (0 if fused else 2)),
        "clocks": sampler.summary(tw0, tw1),
        "device_status": status,
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(name, args.seed, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def gpu_attn_arm(args, rank, world, dist):
    """Attention block of the Nano model: one step = one moe_attention_fwd (projections,
    QK-norm, causal grouped-query attention, output projection with the residual)."""
    import torch

    import aux_loss_free_gb300 as M
    from aux_loss_free_gb300.layer import to_device_bf16

    M.load_library()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    s = ATTN_CONFIGS["attn"]
    H = make_attention(s, "attn", args.seed + rank)
    ms = M.make_attn_shape(s.batch, s.seq, s.d, s.n_head, s.n_kv_head, s.head_dim, s.eps)
    x0 = to_device_bf16(H["x"], dev)
    w_qkv = to_device_bf16(np.concatenate([H["w_q"], H["w_k"], H["w_v"]], axis=0), dev)
    w_o = to_device_bf16(H["w_o"], dev)
    ws = torch.empty(M.moe_attention_workspace_size(ms), dtype=torch.uint8, device=dev)
    out0 = torch.empty(s.T, s.d, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    C = (s.n_head + 2 * s.n_kv_head) * s.head_dim
    qkv = ws[:s.T * C * 2].view(torch.bfloat16).view(s.T, C)   # the workspace's first region
    o_core = torch.empty(s.T, s.n_head * s.head_dim, dtype=torch.bfloat16, device=dev)

    def step(x_in, out):
        M.moe_attention_fwd(ms, x_in, w_qkv, w_o, True, out, ws)

    for _ in range(args.warmup):
        step(x0, out0)
    torch.cuda.synchronize(dev)
    if M.moe_device_status() != 0:
        raise RuntimeError("device status set during warm-up")
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    time.sleep(0.1)
    K = args.steps
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    for i in range(K):
        flush.zero_()
        ev0[i].record(stream)
        step(x0, out0)
        ev1[i].record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    if dist:
        dist.barrier()
    time.sleep(0.05)
    sampler.stop()
    step_ms = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
    total_ms = sum(step_ms)
    if dist:
        t = torch.tensor([total_ms], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    # The attention kernel alone (the block's dominant kernel), on the q, k, v rows the
    # last step left in the workspace, after the same flush.
    core_ms = []
    for i in range(max(3, min(K, 50))):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        M.moe_attention_core(ms, qkv, o_core)
        b.record(stream)
        torch.cuda.synchronize(dev)
        core_ms.append(a.elapsed_time(b))
    status = M.moe_device_status()
    # End to end: tokens in from pinned host memory, the block, the output back, each step.
    Ke = max(3, min(K, 50))
    hx = torch.empty(s.T, s.d, dtype=torch.bfloat16, pin_memory=True)
    hx.copy_(x0.cpu())
    hout = torch.empty(s.T, s.d, dtype=torch.bfloat16, pin_memory=True)
    din = torch.empty_like(x0)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(Ke):
        din.copy_(hx, non_blocking=True)
        step(din, out0)
        hout.copy_(out0, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / Ke
    if rank != 0:
        return
    peaks, peak_note = load_peaks()
    proj, attn, nbytes = attn_algorithmic(s)
    flops = proj + attn
    ms_step = total_ms / K
    roof_s = max(flops / (peaks["bf16_tflops"] * 1e12), nbytes / (peaks["hbm_gbs"] * 1e9))
    core = statistics.median(core_ms)
    core_ach = attn / (core / 1e3) / 1e12
    line = {
        "metric": ATTN_METRIC, "value": world * s.T * K / (total_ms / 1e3), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "attention_block_gqa4_qknorm_B4_S2048", "batch": s.batch, "seq": s.seq, "d": s.d,
                   "n_head": s.n_head, "n_kv_head": s.n_kv_head, "head_dim": s.head_dim, "causal": True,
                   "residual": True, "l2": "512 MiB write before every timed step (L2 129 MB)",
                   "parallelism": f"dp{world}"},
        "layer_roofline": {"flops_per_step": flops, "bytes_per_step": nbytes, "roofline_us": roof_s * 1e6,
                           "measured_us": ms_step * 1e3, "frac": roof_s / (ms_step / 1e3), "peak": peak_note,
                           "bound": "tensor"},
        "roofline": {"kernel": "gqa_attention_kernel (causal attention core)", "bound": "tensor",
                     "achieved": core_ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": core_ach / peaks["bf16_tflops"], "traffic": None,
                     "peak_note": peak_note + " (burst)", "flops_per_launch": attn, "avg_launch_us": core * 1e3},
        "stages_us": {"attention_core": core * 1e3, "projections_qknorm": ms_step * 1e3 - core * 1e3},
        "step_us": {"median": statistics.median(step_ms) * 1e3, "min": min(step_ms) * 1e3,
                    "max": max(step_ms) * 1e3},
        "e2e": {"value": world * s.T / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": int(hx.numel() * 2), "d2h_bytes_per_step": int(hout.numel() * 2),
                "copies": "pinned host buffers on the compute stream"},
        "gpu_launches": K * 5,
        "clocks": sampler.summary(t_wall0, t_wall1),
        "device_status": status,
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = attn_cpu_baseline(args.seed, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def attn_oracle_runner(seed):
    """run(seq) -> seconds for the oracle's attention block on one sequence of `seq` tokens."""
    from oracle import attention_oracle as A

    s = ATTN_CONFIGS["attn"]
    H = make_attention(s, "attn", seed)
    bf = lambda b: f32_from_bf16_bits(b).astype(np.float64)  # noqa: E731
    P = {k: bf(v) for k, v in H.items()}

    def run(seq):
        t0 = time.perf_counter()
        A.gqa_attention(P["x"][:seq], P["w_q"], P["w_k"], P["w_v"], P["w_o"], 1, seq, s.n_head, s.n_kv_head,
                        s.head_dim, s.eps)
        return time.perf_counter() - t0
    return run


def attn_cpu_baseline(seed, seconds):
    if seconds <= 0:
        return None
    run = attn_oracle_runner(seed)
    seq = 512
    run(64)
    done, spent = 0, 0.0
    while spent < seconds and done < 64 * seq:
        spent += run(seq)
        done += seq
    return {"value": done / spent, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{done} tokens as {done // seq} oracle attention blocks of one {seq}-token sequence "
                      f"(fp64 numpy, BLAS on all {cpu_cores()} visible cores), {spent:.1f} s; a shorter "
                      f"sequence than the workload's 2048 (causal cost grows with the sequence)"}


def attn_reference_arm(args, rank, world):
    if rank != 0:
        return
    run = attn_oracle_runner(args.seed)
    seq = 512
    for _ in range(args.warmup):
        run(seq)
    times = [run(seq) for _ in range(args.steps)]
    value = seq * args.steps / sum(times)
    s = ATTN_CONFIGS["attn"]
    line = {"impl": "reference", "metric": ATTN_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "attention_block_gqa4_qknorm_B4_S2048", "batch": s.batch, "seq": s.seq,
                       "d": s.d, "n_head": s.n_head, "n_kv_head": s.n_kv_head, "head_dim": s.head_dim},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "kind": "oracle", "cores": cpu_cores(),
                             "sample": f"each step: the oracle attention block on one {seq}-token sequence"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.cpu_sample_worker:
        # Child of one_thread_baseline: the oracle sample only, printed as JSON.
        print(json.dumps(list(timed_oracle_sample(args.cpu_sample_worker, args.seed, args.cpu_seconds))),
              flush=True)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.gpus != world and world == 1 and args.gpus > 1:
        print(json.dumps({"error": "run N>1 under torch.distributed.run"}), flush=True)
        sys.exit(2)
    if args.impl == "reference":
        (attn_reference_arm if args.workload == "attn" else reference_arm)(args, rank, world)
        return
    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        tdist.init_process_group("nccl")
        dist = tdist
    try:
        arm = gpu_train_arm if args.workload == "train" else (
            gpu_cache_arm if args.workload in CACHE_SLOTS else (gpu_attn_arm if args.workload == "attn" else gpu_arm))
        arm(args, rank, world, dist)
    finally:
        if dist:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
