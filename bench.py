#!/usr/bin/env python3
"""Verify-step benchmark: the W4A16 projection GEMM of the verify block.

Workload (config 1: the 4B-shaped verify step at M = 16, i.e. K = 15 drafts
+ 1): the four W4A16 g128 projections of one decoder layer set (qkv
2560->7680, o 2560->2560, gate_up 2560->19456, down 9728->2560) in one
grouped launch, each step on the weights of another of 36 layers drawn on
the device (1.87 GB, far above L2).

value      = the metric's quantity: W4A16 GEMM algorithmic bytes (packed
             int4 + fp16 group scales + fp16 activations) per step / device
             time per step, GB/s, summed over ranks; K steps timed with CUDA
             events on the launching stream.
roofline   = the same kernel (one grouped launch per step) against the
             measured HBM copy bandwidth, with ncu's DRAM bytes per launch.
verify_step = the whole hot path per step: the layer set, then the int8
             lm_head 2560->151936 with fused greedy argmax and the acceptance
             of 15 seeded drafts in one launch.
e2e        = that whole step through the C ABI with host buffers: one
             cudaMemcpyAsync of the step's inputs from pinned host memory,
             the library's calls (captured as one CUDA graph), one
             cudaMemcpyAsync of the accepted tokens back, host synchronize;
             no torch in the timed loop ("e2e_torch": the same through the
             Python binding).
sweep      = config 2: the 36-layer stack at M in {1,2,4,8,16,21}, as one
             grouped launch for the whole stack and as one per layer set.
cpu_baseline = the CPU oracle on the same layer set.

--impl reference times the oracle alone (the only reference this method has
here) on a bounded sample of the same workload per step.
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

from speculative_decoding_verify_w4a16_gb300 import inputs  # noqa: E402

METRIC = "verify W4A16 GEMM GB/s & % HBM peak at M=16; prefill TFLOP/s at M=8192"
M_VERIFY = 16
K_DRAFT = 15
SEED = 1
COPIES = 3          # projection weight sets rotated per step


def step_bytes(M=M_VERIFY):
    proj = sum(p.N * p.K // 2 + (p.K // 128) * p.N * 2 + M * p.K * 2 for p in inputs.LAYER_PROJS)
    lm = inputs.V_4B * inputs.H_4B + inputs.V_4B * 2 + M * inputs.H_4B * 2
    return proj, lm


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


class _Nvml:
    """Read-only NVML queries through ctypes (SM clock, its maximum, and the
    active clock event reasons); None where the library is missing."""
    SM = 1                                                  # NVML_CLOCK_SM
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, index):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle")
        mx = ctypes.c_uint()
        self.max_mhz = mx.value if self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.SM, ctypes.byref(mx)) == 0 else None

    def sample(self):
        c = self.c
        mhz, rs = c.c_uint(), c.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, self.SM, c.byref(mhz)) != 0:
            return None
        get = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        if get(self.h, c.byref(rs)) != 0:
            return None
        return [str(mhz.value), str(self.max_mhz), ""] + \
            ["Active" if rs.value & bit else "Not Active" for bit in (0x8, 0x40, 0x20, 0x4)]


class ClockSampler:
    """SM clocks and throttle reasons sampled during the timed region: NVML
    every millisecond (the region can be a fraction of a second), else
    nvidia-smi every 200 ms.  The first sample is taken just before the
    timed region starts and the last just after it ends."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.rows = []
        self.source = "nvidia-smi"
        self._stop = threading.Event()
        self._ready = threading.Event()
        self._thr = None
        try:
            self._nvml = _Nvml(index)
            self.source = "nvml"
        except Exception:
            self._nvml = None

    def _run(self):
        while not self._stop.is_set():
            try:
                if self._nvml is not None:
                    row = self._nvml.sample()
                    if row:
                        self.rows.append(row)
                else:
                    out = subprocess.run(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits"], capture_output=True, text=True,
                                         timeout=5).stdout.strip()
                    if out:
                        self.rows.append([x.strip() for x in out.split(",")])
            except Exception:
                pass
            self._ready.set()
            self._stop.wait(0.001 if self._nvml is not None else 0.2)

    def __enter__(self):
        self._thr = threading.Thread(target=self._run, daemon=True)
        self._thr.start()
        self._ready.wait(timeout=10)
        return self

    def __exit__(self, *a):
        self._stop.set()
        self._thr.join(timeout=10)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4)
                          if len(r) > 3 + i and r[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows), "source": self.source}


# --------------------------------------------------------------------- GPU arm
class VerifyStep:
    """Device buffers and the enqueue order of one config-1 verify step."""

    def __init__(self, dev, w4v, torch):
        self.dev, self.w4v, self.torch = dev, w4v, torch
        H, V = inputs.H_4B, inputs.V_4B
        M = M_VERIFY
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        self.host = {}
        self.projs = []
        for c in range(COPIES):
            layer = []
            for p in inputs.LAYER_PROJS:
                q, s = inputs.layer_weights(SEED, c, p)
                if c == 0:
                    self.host[p.name] = (q, s)
                layer.append((p, t(w4v.pack_int4(q)), t(s)))
            self.projs.append(layer)
        # the step's inputs (every projection's activations, the lm_head rows,
        # the drafts) live in one device buffer, so that the end-to-end run
        # moves them with one host -> device copy; likewise the outputs read
        # back (accepted length, emitted tokens) in one buffer
        host_in = [(p.name, inputs.activations(SEED, M, p.K, "bench", p.name)) for p in inputs.LAYER_PROJS]
        host_in.append(("X", inputs.activations(SEED, M, H, "bench", "lm")))
        d = inputs.rng(SEED, "bench-drafts").integers(0, V, size=(1, K_DRAFT)).astype(np.int32)
        host_in.append(("draft", d))
        offs, off = {}, 0
        for name, a in host_in:
            offs[name] = off
            off += (a.nbytes + 255) // 256 * 256
        self.in_host = torch.empty(off, dtype=torch.uint8).pin_memory()
        hv = self.in_host.numpy()
        for name, a in host_in:
            hv[offs[name]:offs[name] + a.nbytes] = np.ascontiguousarray(a).view(np.uint8).reshape(-1)
        self.in_dev = self.in_host.to(dev)

        def view(name, a):
            dt = torch.float16 if a.dtype == np.float16 else torch.int32
            return self.in_dev[offs[name]:offs[name] + a.nbytes].view(dt).view(*a.shape)

        src = dict(host_in)
        self.acts = {p.name: view(p.name, src[p.name]) for p in inputs.LAYER_PROJS}
        self.outs = {p.name: torch.empty((M, p.N), dtype=torch.float16, device=dev) for p in inputs.LAYER_PROJS}
        self.ws = {p.name: w4v.workspace(w4v.w4a16_workspace_bytes(M, p.N, p.K), dev) for p in inputs.LAYER_PROJS}
        W8, s8 = inputs.lmhead_weights(SEED, V, H, "bench")
        self.host["lm"] = (W8, s8)
        self.W8, self.s8 = t(W8), t(s8)
        self.X = view("X", src["X"])
        self.host["acts"] = {k: v.cpu().numpy() for k, v in self.acts.items()}
        self.host["X"] = self.X.cpu().numpy()
        self.tok = torch.empty(M, dtype=torch.int32, device=dev)
        self.ws_lm = w4v.workspace(w4v.w8_lmhead_argmax_workspace_bytes(M, V), dev)
        # drafts: fixed from the seed (the synthetic verify rows do not depend on them)
        self.draft = view("draft", src["draft"])
        self.out_dev = torch.empty(2 + K_DRAFT + 1, dtype=torch.int32, device=dev)
        self.n_acc = self.out_dev[0:1]
        self.out_tok = self.out_dev[2:].view(1, K_DRAFT + 1)
        # one grouped launch per layer set (plan per weight copy)
        self.plans = [w4v.GroupedGemm([(self.acts[p.name], packed, s, None, self.outs[p.name])
                                       for (p, packed, s) in layer]) for layer in self.projs]
        self.launches_per_step = 2

    def enqueue(self, copy):
        self.plans[copy](static_weights=True)
        self.lm_head()

    def lm_head(self):
        """lm_head argmax and acceptance of the drafts, one launch."""
        self.w4v.w8_lmhead_argmax_accept(self.X, self.W8, self.s8, self.draft, out=self.tok, n_out=self.n_acc,
                                         tok_out=self.out_tok, ws=self.ws_lm)


def capture(torch, fn):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


# A kernel's device code: its source and the PTX helpers it inlines (runtime.h,
# also included, holds host-side launch declarations of every kernel family and
# changes whenever one is added).
PROFILES = os.path.join(os.path.dirname(os.path.abspath(__file__)), "profiles")
LM_HEAD_SOURCES = ("w8_lmhead_argmax.cu", "sm103_ptx.cuh")
LM_HEAD_PROFILE = os.path.join(PROFILES, "w8_lmhead_argmax_m16.json")
GEMM_SOURCES = ("w4a16_gemm.cu", "sm103_ptx.cuh")
GEMM_PROFILE = os.path.join(PROFILES, "w4a16_grouped_layer_set_m16.json")


def kernel_source_sha(names):
    """Short fingerprint of the sources a kernel is compiled from."""
    import hashlib
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "speculative_decoding_verify_w4a16_gb300", "csrc")
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(csrc, n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(profile, names):
    """DRAM bytes per launch (read + write) from the committed ncu record of a
    kernel (a small JSON file under profiles/), or None when the record was
    taken from other sources than the ones the kernel is built from now."""
    try:
        with open(profile) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_sha256") != kernel_source_sha(names):
        return None
    try:
        return int(rec["dram_bytes_read"]) + int(rec["dram_bytes_write"])
    except (KeyError, TypeError, ValueError):
        return None


def reduce_step_time(ms_local, world, device=None):
    """Per-step time of the whole job: the maximum over ranks (every rank
    runs the same replica workload; the job ends with the slowest)."""
    if world <= 1:
        return ms_local
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms_local], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(bytes_per_rank, ms_step, world):
    """Whole-job throughput in GB/s: every rank's bytes over the job's step time."""
    return world * bytes_per_rank / (ms_step * 1e-3) / 1e9


def layer_set_bytes(M=M_VERIFY, group=128):
    return sum(p.N * p.K // 2 + (p.K // group) * p.N * 2 + M * p.K * 2 for p in inputs.LAYER_PROJS)


def replay_steps(graph_all, graph_rem, steps, per):
    """Replay a graph of `per` steps (and one of the remainder) for exactly `steps` steps."""
    for _ in range(steps // per):
        graph_all.replay()
    if graph_rem is not None:
        graph_rem.replay()


def run_gpu(args, rank, world):
    import torch
    from speculative_decoding_verify_w4a16_gb300 import _build, w4v
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if rank == 0 or not os.path.exists(_build.LIB):
        _build.build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    w4v.load()
    w4v.init()
    peaks = load_peaks()
    gemm_bytes = layer_set_bytes()

    # ---- config 1: the layer set at M = 16, one grouped launch per step, each
    # step on the weights of another of 36 layers (1.87 GB, far above L2)
    stack = Stack(dev, w4v, torch)
    sets = stack.layer_plans(M_VERIFY)
    L = stack.LAYERS
    for i in range(max(args.warmup, 3)):
        sets[i % L](static_weights=True)
    torch.cuda.synchronize()
    g_all = capture(torch, lambda: [sets[i](static_weights=True) for i in range(L)])
    rem = args.steps % L
    g_rem = capture(torch, lambda: [sets[i](static_weights=True) for i in range(rem)]) if rem else None
    replay_steps(g_all, None, max(args.warmup, 3) * L, L)
    torch.cuda.synchronize()

    # ---- timed region: exactly K steps, no host synchronisation inside -------
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        start.record()
        replay_steps(g_all, g_rem, args.steps, L)
        end.record()
        torch.cuda.synchronize()
    ms_total = start.elapsed_time(end)
    ms_step = reduce_step_time(ms_total / args.steps, world, dev)
    value = job_value(gemm_bytes, ms_step, world)
    gemm_gbs = gemm_bytes / (ms_step * 1e-3) / 1e9
    del g_all, g_rem
    check_device_status(w4v, "layer set")

    # ---- the whole verify step: layer set + lm_head argmax + acceptance -------
    step = VerifyStep(dev, w4v, torch)
    proj_bytes, lm_bytes = step_bytes()
    for i in range(3):
        step.enqueue(i % COPIES)
    torch.cuda.synchronize()
    reps = 20
    step_ms = time_graph(torch, lambda: [step.enqueue(i % COPIES) for i in range(reps)]) / reps
    lm_ms = time_graph(torch, lambda: [step.lm_head() for _ in range(reps)]) / reps
    lm_gbs = lm_bytes / (lm_ms * 1e-3) / 1e9
    verify_step = {"ms": round(step_ms, 5), "bytes": proj_bytes + lm_bytes,
                   "GB/s": round((proj_bytes + lm_bytes) / (step_ms * 1e-3) / 1e9, 1),
                   "launches": step.launches_per_step,
                   "what": "grouped W4A16 layer set (3 rotating weight copies) + fused int8 lm_head argmax and "
                           "acceptance of 15 drafts, %d steps in one CUDA graph" % reps,
                   "lm_head": {"ms": round(lm_ms, 5), "bytes": lm_bytes, "GB/s": round(lm_gbs, 1),
                               "frac": round(lm_gbs / peaks["hbm_gbs"], 4),
                               "traffic": profiled_traffic(LM_HEAD_PROFILE, LM_HEAD_SOURCES)}}
    check_device_status(w4v, "verify step")

    # ---- per projection, one launch each (each launch on another layer) ------
    kern = {}
    for p in inputs.LAYER_PROJS:
        ms = stack.time_projection(p, M_VERIFY)
        b = p.N * p.K // 2 + (p.K // 128) * p.N * 2 + M_VERIFY * p.K * 2
        gbs = b / (ms * 1e-3) / 1e9
        kern[p.name] = {"ms": round(ms, 5), "bytes": b, "GB/s": round(gbs, 1), "frac": round(gbs / peaks["hbm_gbs"], 4)}
    single_ms = sum(kern[p.name]["ms"] for p in inputs.LAYER_PROJS)
    check_device_status(w4v, "per-projection launches")

    # ---- end to end through the C ABI with host buffers ------------------------
    e2e = run_e2e_capi(args, step, w4v, torch, proj_bytes + lm_bytes, gemm_bytes, world)
    check_device_status(w4v, "end to end (C ABI)")
    e2e_torch = run_e2e(args, step, torch, proj_bytes + lm_bytes, world)
    check_device_status(w4v, "end to end (binding)")

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic",
        "config": {"workload": "cfg1: 4B-shaped W4A16 g128 layer set (qkv 2560->7680, o 2560->2560, gate_up "
                               "2560->19456, down 9728->2560) at M=16 (K=15 drafts + 1), one grouped launch per step",
                   "M": M_VERIFY, "K_draft": K_DRAFT, "bytes_per_step": gemm_bytes,
                   "l2": "inputs larger than L2: each step reads another of 36 layers' weights (1.87 GB in all)",
                   "graph": "36 steps per CUDA graph (the remainder in a second graph)",
                   "parallelism": "replicas" if world > 1 else "1 GPU",
                   "weights": "static (W4V_STATIC_WEIGHTS: weights may be loaded before the previous kernel ends; "
                              "activations and outputs wait for it)"},
        "roofline": {"bound": "hbm", "kernel": "w4a16_decode_kernel (grouped launch of the layer set, M=16)",
                     "achieved": round(gemm_gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(gemm_gbs / peaks["hbm_gbs"], 4),
                     "traffic": profiled_traffic(GEMM_PROFILE, GEMM_SOURCES),
                     "traffic_source": "dram__bytes_read.sum + dram__bytes_write.sum per launch, ncu record "
                                       "profiles/w4a16_grouped_layer_set_m16.json (null if taken from other sources)",
                     "algorithmic_bytes": gemm_bytes,
                     "timing": "CUDA events on the launching stream around the K timed steps",
                     "peak_source": peaks["source"] + " (hbm copy, burst)"},
        "verify_step": verify_step,
        "gemm_m16_single_launches": {"ms": round(single_ms, 5), "GB/s": round(gemm_bytes / (single_ms * 1e-3) / 1e9, 1),
                                     "frac": round(gemm_bytes / (single_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                                     "per_projection": kern},
        "e2e": e2e,
        "e2e_torch": e2e_torch,
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
    }
    if args.sweep:
        result["sweep"] = stack.sweep(peaks)
        check_device_status(w4v, "36-layer sweep")
        result["verify_36_layers"] = stack.full_verify(step.W8, step.s8, peaks)
        check_device_status(w4v, "36-layer verify")
        # a 4-bit g128 drafter of the pages' size (277 MB): five layer sets, 263 MB
        drafter = Stack(dev, w4v, torch, group=128, layers=5)
        result["drafter_5_layers"] = drafter.stack_graph(peaks)
        check_device_status(w4v, "drafter stack")
        del drafter
        # the same kernel's streaming rate: one 200 MB projection (N = 155648,
        # K = 2560) at M = 16, where the launch's ramp and tail are amortised
        result["gemm_m16_streaming"] = run_streaming(dev, w4v, torch, peaks)
        check_device_status(w4v, "streaming")
        # the group-size-32 W4A16 target (compressed-tensors format), same shapes
        g32 = Stack(dev, w4v, torch, group=32)
        result["gemm_m16_g32"] = g32.layer_set(peaks)
        check_device_status(w4v, "group-32 layer set")
        del g32
    del stack, sets
    torch.cuda.empty_cache()
    if args.prefill:
        result["prefill"] = run_prefill(dev, w4v, torch, peaks)
        check_device_status(w4v, "prefill")
        result["lmhead_batched"] = run_lmhead_batched(dev, w4v, torch, peaks)
        check_device_status(w4v, "batched lm_head")
    result["ngram_draft"] = run_ngram(dev, w4v, torch)
    result["gdn_state"] = run_gdn(dev, w4v, torch)
    check_device_status(w4v, "drafter and recurrent state")
    if rank == 0 and not args.no_cpu:
        result["cpu_baseline"] = cpu_baseline(step)
    return result


def check_device_status(w4v, leg="bench"):
    """A kernel that gave up a bounded wait leaves its status word set (read and
    cleared here) and its outputs and timings meaningless: fail loudly instead
    of printing them."""
    st = w4v.get_status()
    if st != 0:
        raise RuntimeError("device status %d after the %s leg: a kernel gave up a bounded wait; "
                           "the measurements are invalid" % (st, leg))


def run_e2e(args, step, torch, total_bytes, world):
    """Host buffers in, accepted tokens out, through the same calls, one graph per step."""
    h_out = torch.empty(step.out_dev.numel(), dtype=torch.int32).pin_memory()
    h_n = h_out[0:1]

    def body(c):
        step.in_dev.copy_(step.in_host, non_blocking=True)     # all of the step's inputs
        step.enqueue(c)
        h_out.copy_(step.out_dev, non_blocking=True)           # accepted length + emitted tokens

    for c in range(COPIES):
        body(c)
    torch.cuda.synchronize()
    graphs = [capture(torch, lambda c=c: body(c)) for c in range(COPIES)]
    for c in range(COPIES):
        graphs[c].replay()
    torch.cuda.synchronize()
    steps = args.steps
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for i in range(steps):
        graphs[i % COPIES].replay()
        torch.cuda.current_stream().synchronize()     # the host reads the accepted tokens every step
        _ = int(h_n[0])
    ms = reduce_step_time((time.perf_counter() - t0) / steps * 1e3, world, step.draft.device)
    h2d = step.in_host.numel()
    d2h = h_out.numel() * 4
    return {"value": round(job_value(layer_set_bytes(), ms, world), 1), "unit": "GB/s",
            "ms_per_step": round(ms, 5), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "whole_step_GB/s": round(job_value(total_bytes, ms, world), 1),
            "how": "through the Python binding: one pinned host -> device copy of all activations and drafts, "
                   "one CUDA graph of the step, one device -> host copy of the accepted length and tokens, "
                   "host synchronize each step (wall clock)"}


def _cudart():
    """The CUDA runtime library (for the C-ABI end-to-end leg)."""
    import ctypes
    import ctypes.util
    for cand in (ctypes.util.find_library("cudart"), "/usr/local/cuda/lib64/libcudart.so", "libcudart.so.13"):
        if not cand:
            continue
        try:
            return ctypes.CDLL(cand)
        except OSError:
            continue
    raise RuntimeError("libcudart not found")


def run_e2e_capi(args, step, w4v, torch, total_bytes, gemm_bytes, world):
    """The whole verify step end to end through the C ABI with host buffers and
    no torch in the timed loop: per step one cudaMemcpyAsync of all the step's
    inputs (activations of the four projections and the lm_head, drafts) from
    pinned host memory, the grouped W4A16 launch and the fused lm_head argmax +
    acceptance (libw4v's C entry points), one cudaMemcpyAsync of the accepted
    length and tokens back, all captured once as a CUDA graph per weight copy;
    the host launches the graph, polls the stream until the step completes and
    reads the accepted length."""
    import ctypes
    cu = _cudart()
    lib = w4v.load()
    P, S = ctypes.c_void_p, ctypes.c_size_t
    cu.cudaStreamCreateWithFlags.argtypes = [ctypes.POINTER(P), ctypes.c_uint]
    cu.cudaHostAlloc.argtypes = [ctypes.POINTER(P), S, ctypes.c_uint]
    cu.cudaFreeHost.argtypes = [P]
    cu.cudaMemcpyAsync.argtypes = [P, P, S, ctypes.c_int, P]
    cu.cudaStreamBeginCapture.argtypes = [P, ctypes.c_int]
    cu.cudaStreamEndCapture.argtypes = [P, ctypes.POINTER(P)]
    cu.cudaGraphInstantiate.argtypes = [ctypes.POINTER(P), P, ctypes.c_ulonglong]
    cu.cudaGraphLaunch.argtypes = [P, P]
    cu.cudaStreamSynchronize.argtypes = [P]
    cu.cudaStreamQuery.argtypes = [P]
    cu.cudaGraphExecDestroy.argtypes = [P]
    cu.cudaGraphDestroy.argtypes = [P]
    cu.cudaStreamDestroy.argtypes = [P]

    def ok(code, what):
        if code != 0:
            raise RuntimeError("%s failed with CUDA error %d" % (what, code))

    stream = P()
    ok(cu.cudaStreamCreateWithFlags(ctypes.byref(stream), 1), "cudaStreamCreateWithFlags")
    n_in = step.in_host.numel()
    n_out = step.out_dev.numel() * 4
    h_in, h_out = P(), P()
    ok(cu.cudaHostAlloc(ctypes.byref(h_in), n_in, 0), "cudaHostAlloc")
    ok(cu.cudaHostAlloc(ctypes.byref(h_out), n_out, 0), "cudaHostAlloc")
    ctypes.memmove(h_in, step.in_host.data_ptr(), n_in)
    V, H = inputs.V_4B, inputs.H_4B
    execs, graphs = [], []
    for c in range(COPIES):
        plan = step.plans[c]
        ok(cu.cudaStreamBeginCapture(stream, 2), "cudaStreamBeginCapture")     # relaxed mode
        ok(cu.cudaMemcpyAsync(P(step.in_dev.data_ptr()), h_in, n_in, 1, stream), "cudaMemcpyAsync in")
        st = lib.w4a16_gemm_grouped(ctypes.byref(plan.handle), P(plan.ws.data_ptr()), plan.ws.numel(),
                                    w4v.STATIC_WEIGHTS, stream)
        st2 = lib.w8_lmhead_argmax_accept(P(step.X.data_ptr()), P(step.W8.data_ptr()), P(step.s8.data_ptr()),
                                          1, K_DRAFT, H, V, P(step.draft.data_ptr()), P(step.tok.data_ptr()),
                                          P(step.n_acc.data_ptr()), P(step.out_tok.data_ptr()), None,
                                          P(step.ws_lm.data_ptr()), step.ws_lm.numel(), stream)
        ok(cu.cudaMemcpyAsync(h_out, P(step.out_dev.data_ptr()), n_out, 2, stream), "cudaMemcpyAsync out")
        g = P()
        ok(cu.cudaStreamEndCapture(stream, ctypes.byref(g)), "cudaStreamEndCapture")
        if st != 0 or st2 != 0:
            raise RuntimeError("library call failed during capture: %d %d" % (st, st2))
        ex = P()
        ok(cu.cudaGraphInstantiate(ctypes.byref(ex), g, 0), "cudaGraphInstantiate")
        graphs.append(g)
        execs.append(ex)
    n_acc = ctypes.cast(h_out, ctypes.POINTER(ctypes.c_int32))
    for i in range(max(args.warmup, 3)):
        ok(cu.cudaGraphLaunch(execs[i % COPIES], stream), "cudaGraphLaunch")
        ok(cu.cudaStreamSynchronize(stream), "cudaStreamSynchronize")
    if world > 1:
        torch.distributed.barrier()
    # The host waits for each step by polling the stream (a serving loop's
    # low-latency wait: no thread wake-up on completion), then reads the result.
    launch, query = cu.cudaGraphLaunch, cu.cudaStreamQuery
    t0 = time.perf_counter()
    acc = 0
    for i in range(args.steps):
        launch(execs[i % COPIES], stream)
        while True:
            q = query(stream)
            if q == 0:
                break
            if q != 600:                     # cudaErrorNotReady: still running
                raise RuntimeError("cudaStreamQuery failed with CUDA error %d" % q)
        acc += n_acc[0]                      # the host reads the accepted length every step
    ms = reduce_step_time((time.perf_counter() - t0) / args.steps * 1e3, world, step.draft.device)
    for ex, g in zip(execs, graphs):
        cu.cudaGraphExecDestroy(ex)
        cu.cudaGraphDestroy(g)
    cu.cudaFreeHost(h_in)
    cu.cudaFreeHost(h_out)
    cu.cudaStreamDestroy(stream)
    return {"value": round(job_value(gemm_bytes, ms, world), 1), "unit": "GB/s", "ms_per_step": round(ms, 5),
            "h2d_bytes_per_step": int(n_in), "d2h_bytes_per_step": int(n_out),
            "whole_step_GB/s": round(job_value(total_bytes, ms, world), 1),
            "how": "C ABI through ctypes and the CUDA runtime, no torch in the loop: per step one CUDA graph "
                   "(cudaMemcpyAsync of the inputs from pinned host memory, w4a16_gemm_grouped, "
                   "w8_lmhead_argmax_accept, cudaMemcpyAsync of the accepted tokens back), then "
                   "cudaStreamQuery polled until the step completes and a host read of the accepted length "
                   "(wall clock); value = the "
                   "W4A16 GEMM bytes of the step over the step's end-to-end time"}


def time_graph(torch, fn, reps=3):
    """Device ms of one replay of a graph of fn, median of reps timed replays."""
    fn()
    torch.cuda.synchronize()
    g = capture(torch, fn)
    g.replay()
    torch.cuda.synchronize()
    out = []
    for _ in range(reps):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        g.replay()
        e.record()
        torch.cuda.synchronize()
        out.append(s.elapsed_time(e))
    del g
    return statistics.median(out)


class Stack:
    """36-layer stack of the projections (config 2), weights drawn on the device
    directly in packed form (uniform random bytes = uniform iid 4-bit codes in
    any nibble order), fp16 scales U[0.005, 0.02]: 1.87 GB, far above L2, so
    every launch streams its weights from HBM."""

    LAYERS = 36

    def __init__(self, dev, w4v, torch, group=128, layers=LAYERS):
        self.dev, self.w4v, self.torch = dev, w4v, torch
        self.group = group
        self.LAYERS = layers
        g = torch.Generator(device=dev)
        g.manual_seed(SEED + group)
        self.g = g
        self.layers = []
        for _ in range(self.LAYERS):
            lay = []
            for p in inputs.LAYER_PROJS:
                packed = torch.randint(0, 256, (w4v.packed_bytes(p.N, p.K),), generator=g, device=dev,
                                       dtype=torch.uint8)
                sc = (torch.rand(((p.K // group), p.N), generator=g, device=dev) * 0.015 + 0.005).half()
                lay.append((p, packed, sc))
            self.layers.append(lay)

    def proj_bytes(self, p, M):
        return p.N * p.K // 2 + (p.K // self.group) * p.N * 2 + M * p.K * 2

    def _buffers(self, M):
        torch = self.torch
        acts = {p.name: torch.randn((M, p.K), generator=self.g, device=self.dev).half() for p in inputs.LAYER_PROJS}
        outs = {p.name: torch.empty((M, p.N), device=self.dev, dtype=torch.float16) for p in inputs.LAYER_PROJS}
        wss = {p.name: self.w4v.workspace(self.w4v.w4a16_workspace_bytes(M, p.N, p.K), self.dev)
               for p in inputs.LAYER_PROJS}
        return acts, outs, wss

    def time_projection(self, proj, M):
        """ms per launch of one projection, launched once per layer (36 launches)."""
        acts, outs, wss = self._buffers(M)
        k = [i for i, p in enumerate(inputs.LAYER_PROJS) if p.name == proj.name][0]

        def run():
            for lay in self.layers:
                p, packed, sc = lay[k]
                self.w4v.w4a16_gemm(acts[p.name], packed, sc, p.N, out=outs[p.name], ws=wss[p.name],
                                    static_weights=True, group=self.group)

        return time_graph(self.torch, run) / self.LAYERS

    def layer_plans(self, M, bufs=None):
        """One grouped plan per layer: its four projections in one launch."""
        acts, outs, _ = bufs if bufs is not None else self._buffers(M)
        return [self.w4v.GroupedGemm([(acts[p.name], packed, sc, None, outs[p.name]) for (p, packed, sc) in lay],
                                     group=self.group) for lay in self.layers]

    def stack_plan(self, M, bufs=None):
        """The whole stack (every projection of every layer) as one grouped launch."""
        acts, outs, _ = bufs if bufs is not None else self._buffers(M)
        return self.w4v.GroupedGemm([(acts[p.name], packed, sc, None, outs[p.name])
                                     for lay in self.layers for (p, packed, sc) in lay], group=self.group)

    def bytes(self, M):
        return self.LAYERS * sum(self.proj_bytes(p, M) for p in inputs.LAYER_PROJS)

    def layer_set(self, peaks, M=M_VERIFY):
        """The layer set in one grouped launch per layer (36 launches, one graph),
        and per projection one launch each."""
        plans = self.layer_plans(M)
        ms = time_graph(self.torch, lambda: [g(static_weights=True) for g in plans]) / self.LAYERS
        b = sum(self.proj_bytes(p, M) for p in inputs.LAYER_PROJS)
        gbs = b / (ms * 1e-3) / 1e9
        per = {}
        for p in inputs.LAYER_PROJS:
            pm = self.time_projection(p, M)
            per[p.name] = {"ms": round(pm, 5), "GB/s": round(self.proj_bytes(p, M) / (pm * 1e-3) / 1e9, 1)}
        return {"group": self.group, "M": M, "ms": round(ms, 5), "bytes": b, "GB/s": round(gbs, 1),
                "frac": round(gbs / peaks["hbm_gbs"], 4), "launch": "one grouped launch per layer set",
                "single_launches_per_projection": per}

    def stack_graph(self, peaks, M=M_VERIFY):
        """Every projection of every layer in one grouped launch."""
        big = self.stack_plan(M)
        ms = time_graph(self.torch, lambda: [big(static_weights=True) for _ in range(3)]) / 3
        b = self.bytes(M)
        gbs = b / (ms * 1e-3) / 1e9
        return {"layers": self.LAYERS, "group": self.group, "M": M, "ms": round(ms, 4), "bytes": b,
                "GB/s": round(gbs, 1), "frac": round(gbs / peaks["hbm_gbs"], 4), "launches": 1}

    def sweep(self, peaks):
        """Config 2: the 36-layer stack at each verify size, as one grouped launch
        for the whole stack, as one grouped launch per layer set, and as one
        launch per projection."""
        out = {}
        for M in (1, 2, 4, 8, 16, 21):
            bufs = self._buffers(M)
            acts, outs, wss = bufs
            b = self.bytes(M)
            big = self.stack_plan(M, bufs)
            ms_big = time_graph(self.torch, lambda: [big(static_weights=True) for _ in range(3)]) / 3
            plans = self.layer_plans(M, bufs)
            ms_lay = time_graph(self.torch, lambda: [g(static_weights=True) for g in plans])

            def run():
                for lay in self.layers:
                    for (p, packed, sc) in lay:
                        self.w4v.w4a16_gemm(acts[p.name], packed, sc, p.N, out=outs[p.name], ws=wss[p.name],
                                            static_weights=True)

            ms_one = time_graph(self.torch, run)
            f = lambda ms: round(b / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)
            out["M=%d" % M] = {"ms": round(ms_big, 4), "GB/s": round(b / (ms_big * 1e-3) / 1e9, 1),
                               "frac": f(ms_big), "launches": 1,
                               "per_layer_set": {"ms": round(ms_lay, 4), "frac": f(ms_lay), "launches": self.LAYERS},
                               "per_projection": {"ms": round(ms_one, 4), "frac": f(ms_one),
                                                  "launches": 4 * self.LAYERS}}
            del big, plans
        return out

    def full_verify(self, W8, s8, peaks):
        """The whole 36-layer verify step as one CUDA graph: one grouped launch per
        layer set (the layers of a model run one after the other), then the
        lm_head argmax with acceptance of M-1 drafts in one launch (M = 16:
        K = 15; M = 21: K = 20 with seeded -1 padding)."""
        torch, w4v = self.torch, self.w4v
        H, V = inputs.H_4B, inputs.V_4B
        out = {}
        for M in (16, 21):
            plans = self.layer_plans(M)
            X = torch.randn((M, H), generator=self.g, device=self.dev).half()
            d = inputs.rng(SEED, "stack-drafts", M).integers(0, V, size=(1, M - 1)).astype(np.int32)
            if M == 21:
                d[0, 12:] = -1
            d = torch.from_numpy(d).to(self.dev)
            tok = torch.empty(M, dtype=torch.int32, device=self.dev)
            n = torch.empty(1, dtype=torch.int32, device=self.dev)
            o = torch.empty((1, M), dtype=torch.int32, device=self.dev)
            ws = w4v.workspace(w4v.w8_lmhead_argmax_workspace_bytes(M, V), self.dev)

            def run():
                for g in plans:
                    g(static_weights=True)
                w4v.w8_lmhead_argmax_accept(X, W8, s8, d, out=tok, n_out=n, tok_out=o, ws=ws)

            ms = time_graph(torch, run)
            b = self.bytes(M) + V * H + 2 * V + 2 * M * H
            gbs = b / (ms * 1e-3) / 1e9
            out["M=%d" % M] = {"ms": round(ms, 4), "GB/s": round(gbs, 1), "frac": round(gbs / peaks["hbm_gbs"], 4),
                               "launches": self.LAYERS + 1, "K_draft": M - 1}
            del plans
        return out


def run_streaming(dev, w4v, torch, peaks):
    """Steady-state rate of the verify-sized GEMM on one large weight matrix."""
    N, K, M = 155648, 2560, M_VERIFY
    g = torch.Generator(device=dev)
    g.manual_seed(SEED + 3)
    packs = [torch.randint(0, 256, (w4v.packed_bytes(N, K),), generator=g, device=dev, dtype=torch.uint8)
             for _ in range(2)]
    sc = (torch.rand(((K // 128), N), generator=g, device=dev) * 0.015 + 0.005).half()
    A = torch.randn((M, K), generator=g, device=dev).half()
    C = torch.empty((M, N), device=dev, dtype=torch.float16)
    ws = w4v.workspace(w4v.w4a16_workspace_bytes(M, N, K), dev)
    ms = time_graph(torch, lambda: [w4v.w4a16_gemm(A, packs[i % 2], sc, N, out=C, ws=ws, static_weights=True)
                                    for i in range(10)]) / 10
    b = N * K // 2 + (K // 128) * N * 2 + M * K * 2
    gbs = b / (ms * 1e-3) / 1e9
    return {"N": N, "K": K, "M": M, "ms": round(ms, 5), "bytes": b, "GB/s": round(gbs, 1),
            "frac": round(gbs / peaks["hbm_gbs"], 4)}


def run_prefill(dev, w4v, torch, peaks):
    """The layer set at prefill sizes (M = 2048 and 8192): tensor-bound."""
    g = torch.Generator(device=dev)
    g.manual_seed(SEED + 7)
    out = {}
    for M in (8192, 2048):
        projs = []
        for p in inputs.LAYER_PROJS:
            packed = torch.randint(0, 256, (w4v.packed_bytes(p.N, p.K),), generator=g, device=dev, dtype=torch.uint8)
            sc = (torch.rand(((p.K // 128), p.N), generator=g, device=dev) * 0.015 + 0.005).half()
            A = torch.randn((M, p.K), generator=g, device=dev).half()
            C = torch.empty((M, p.N), device=dev, dtype=torch.float16)
            ws = w4v.workspace(w4v.w4a16_workspace_bytes(M, p.N, p.K), dev)
            projs.append((p, packed, sc, A, C, ws))

        def run():
            for (p, packed, sc, A, C, ws) in projs:
                w4v.w4a16_gemm(A, packed, sc, p.N, out=C, ws=ws)

        per = {}
        for (p, packed, sc, A, C, ws) in projs:
            ms = time_graph(torch, lambda p=p, packed=packed, sc=sc, A=A, C=C, ws=ws:
                            w4v.w4a16_gemm(A, packed, sc, p.N, out=C, ws=ws))
            per[p.name] = round(2.0 * M * p.N * p.K / (ms * 1e-3) / 1e12, 1)
        ms = time_graph(torch, run)
        flop = sum(2.0 * M * p.N * p.K for p in inputs.LAYER_PROJS)
        tf = flop / (ms * 1e-3) / 1e12
        out["M=%d" % M] = {"bound": "tensor", "ms": round(ms, 4), "achieved": round(tf, 1), "unit": "TFLOP/s",
                           "peak": peaks["bf16_tflops"], "frac": round(tf / peaks["bf16_tflops"], 4),
                           "peak_source": peaks["source"] + " (dense bf16 = fp16 rate, burst)",
                           "per_projection_TFLOP/s": per}
        del projs
        torch.cuda.empty_cache()
    return out


def run_lmhead_batched(dev, w4v, torch, peaks):
    """Batched verify of 8 sequences x 16 positions (M = 128) through the int8
    lm_head with per-sequence acceptance, and the prefill's last-row lm_head."""
    H, V = inputs.H_4B, inputs.V_4B
    W8, s8 = inputs.lmhead_weights(SEED, V, H, "bench")
    Wd = torch.from_numpy(W8).to(dev)
    sd = torch.from_numpy(s8).to(dev)
    out = {}
    for (B, K1) in ((8, 16), (1, 1)):
        M = B * K1
        X = torch.from_numpy(inputs.activations(SEED, M, H, "lmb")).to(dev)
        tok = torch.empty(M, dtype=torch.int32, device=dev)
        ws = w4v.workspace(w4v.w8_lmhead_argmax_workspace_bytes(M, V), dev)
        d = torch.from_numpy(inputs.rng(SEED, "lmb-d").integers(0, V, size=(B, K1 - 1)).astype(np.int32)).to(dev)
        n = torch.empty(B, dtype=torch.int32, device=dev)
        o = torch.empty((B, K1), dtype=torch.int32, device=dev)

        def step():
            w4v.w8_lmhead_argmax_accept(X, Wd, sd, d, out=tok, n_out=n, tok_out=o, ws=ws)

        ms = time_graph(torch, lambda: [step() for _ in range(10)]) / 10
        b = V * H + 2 * V + 2 * M * H
        gbs = b / (ms * 1e-3) / 1e9
        out["M=%d" % M] = {"ms": round(ms, 5), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 4),
                           "TFLOP/s": round(2.0 * M * V * H / (ms * 1e-3) / 1e12, 1),
                           "workload": "%d sequences x %d positions + acceptance" % (B, K1)}
    return out


def run_ngram(dev, w4v, torch):
    """Prompt-lookup drafting of K = 23 tokens (the n-gram entry's K) for 8
    prompt-like contexts of 4096 tokens, and for one 64K-token context."""
    out = {}
    for (B, ld) in ((8, 4096), (1, 65536)):
        ctx, lens = inputs.ngram_contexts(SEED, B, ld, inputs.V_4B, "bench", ragged=False)
        c = torch.from_numpy(ctx).to(dev)
        l = torch.from_numpy(lens).to(dev)
        d = torch.empty((B, 23), dtype=torch.int32, device=dev)
        m = torch.empty(B, dtype=torch.int32, device=dev)
        ws = w4v.workspace(w4v.load().ngram_draft_workspace_bytes(B), dev)
        ms = time_graph(torch, lambda: [w4v.ngram_draft(c, l, 1, 4, 23, out=d, match=m, ws=ws)
                                        for _ in range(20)]) / 20
        out["B=%d,L=%d" % (B, ld)] = {"us": round(ms * 1e3, 2), "n_min": 1, "n_max": 4, "K": 23,
                                      "GB/s": round(B * ld * 4 / (ms * 1e-3) / 1e9, 1)}
    return out


def run_gdn(dev, w4v, torch):
    """Recurrent-state handling of one Gated DeltaNet layer across a verify
    block of 16 positions: gdn_verify (outputs, state read) then gdn_commit
    (replay of the accepted prefix, state written), and gdn_step (the
    previous block's commit and this block's verify in one launch), assumed
    head shape 32 heads x 128 x 128, for 1 and 8 sequences."""
    out = {}
    H, d, T = 32, 128, 16
    g = torch.Generator(device=dev)
    g.manual_seed(SEED)
    for B in (1, 8):
        S = torch.randn((B, H, d, d), generator=g, device=dev)
        q = torch.nn.functional.normalize(torch.randn((B, T, H, d), generator=g, device=dev), dim=-1).half()
        k = torch.nn.functional.normalize(torch.randn((B, T, H, d), generator=g, device=dev), dim=-1).half()
        v = torch.randn((B, T, H, d), generator=g, device=dev).half()
        a = torch.rand((B, T, H), generator=g, device=dev) * 0.5 + 0.5
        be = torch.rand((B, T, H), generator=g, device=dev)
        n = torch.full((B,), T - 1, dtype=torch.int32, device=dev)
        o = torch.empty((B, T, H, d), dtype=torch.float16, device=dev)

        def step():
            w4v.gdn_verify(S, q, k, v, a, be, out=o)
            w4v.gdn_commit(S, k, v, a, be, n)

        def fused():
            # the previous block's commit and this block's verify in one launch
            w4v.gdn_step(S, (k, v, a, be, n), q, k, v, a, be, out=o)

        ms = time_graph(torch, lambda: [step() for _ in range(20)]) / 20
        ms_f = time_graph(torch, lambda: [fused() for _ in range(20)]) / 20
        state_bytes = 3 * B * H * d * d * 4          # verify read, commit read + write
        out["B=%d" % B] = {"us": round(ms * 1e3, 2), "T": T, "heads": H, "dk": d, "dv": d,
                           "state_GB/s": round(state_bytes / (ms * 1e-3) / 1e9, 1),
                           "step_us": round(ms_f * 1e3, 2),
                           "step_state_GB/s": round(2 * B * H * d * d * 4 / (ms_f * 1e-3) / 1e9, 1)}
    return out


# --------------------------------------------------------------------- CPU arm
def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def oracle_gemm(host, frac=1.0):
    """The oracle on the config-1 layer set (the metric's quantity); frac < 1
    keeps that fraction of every weight matrix's output rows (all 16
    activation rows, full K).  Returns the algorithmic bytes it processed."""
    import oracle
    nbytes = 0
    for p in inputs.LAYER_PROJS:
        q, s = host[p.name]
        n = max(8, int(p.N * frac) // 8 * 8)
        A = host["acts"][p.name]
        oracle.w4a16_gemm(A, q[:n], np.ascontiguousarray(s[:, :n]))
        nbytes += n * p.K // 2 + (p.K // 128) * n * 2 + M_VERIFY * p.K * 2
    return nbytes


def oracle_step(host, frac=1.0):
    """The oracle on the whole config-1 step: the layer set, then the lm_head,
    argmax and acceptance (same sampling).  Returns the bytes processed."""
    import oracle
    nbytes = oracle_gemm(host, frac)
    W8, s8 = host["lm"]
    v = max(8, int(W8.shape[0] * frac))
    L = oracle.lmhead_logits(host["X"], W8[:v], s8[:v])
    t = oracle.argmax(L)
    d = np.zeros((1, K_DRAFT), np.int32)
    oracle.spec_accept(t.reshape(1, -1), d)
    nbytes += v * inputs.H_4B + v * 2 + M_VERIFY * inputs.H_4B * 2
    return nbytes


def cpu_baseline(step):
    import oracle
    oracle.build()
    threads = oracle.num_threads()
    # the full layer set, repeated for about 10 s of CPU work (at most 64 times)
    reps, nbytes = 0, 0
    t0 = time.perf_counter()
    while reps < 64 and (reps == 0 or time.perf_counter() - t0 < 10.0):
        nbytes += oracle_gemm(step.host, 1.0)
        reps += 1
    dt = time.perf_counter() - t0
    t0 = time.perf_counter()
    nbytes_step = oracle_step(step.host, 1.0)
    dt_step = time.perf_counter() - t0
    # the same oracle on one thread, on 1/16 of every matrix's output rows
    oracle.set_num_threads(1)
    try:
        t1 = time.perf_counter()
        nb1 = oracle_gemm(step.host, 1.0 / 16)
        dt1 = time.perf_counter() - t1
    finally:
        oracle.set_num_threads(threads)
    # the projections' dequantization and GEMM timed apart (all threads)
    t_deq = t_mm = 0.0
    for p in inputs.LAYER_PROJS:
        q, sc = step.host[p.name]
        t2 = time.perf_counter()
        w = oracle.dequant_w4(q, sc)
        t3 = time.perf_counter()
        oracle.matmul_dequantized(step.host["acts"][p.name], w)
        t4 = time.perf_counter()
        t_deq += t3 - t2
        t_mm += t4 - t3
    return {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": "the full cfg1 W4A16 layer set (4 projections, M=16), double precision, OpenMP over "
                      "output rows, %d times back to back" % reps, "repetitions": reps,
            "affinity_cores": _cores(), "nproc": os.cpu_count(),
            "whole_step": {"GB/s": round(nbytes_step / dt_step / 1e9, 4), "seconds": round(dt_step, 2),
                           "sample": "layer set + lm_head + argmax + acceptance"},
            "single_thread": {"GB/s": round(nb1 / dt1 / 1e9, 4), "seconds": round(dt1, 2),
                              "sample": "1/16 of every matrix's output rows, one thread"},
            "projections_split_s": {"dequant": round(t_deq, 3), "gemm": round(t_mm, 3)}}


def host_inputs():
    host = {}
    for p in inputs.LAYER_PROJS:
        host[p.name] = inputs.layer_weights(SEED, 0, p)
    host["acts"] = {p.name: inputs.activations(SEED, M_VERIFY, p.K, "bench", p.name) for p in inputs.LAYER_PROJS}
    host["lm"] = inputs.lmhead_weights(SEED, inputs.V_4B, inputs.H_4B, "bench")
    host["X"] = inputs.activations(SEED, M_VERIFY, inputs.H_4B, "bench", "lm")
    return host


def run_reference(args, rank, world):
    import oracle
    oracle.build()
    host = host_inputs()
    frac = args.ref_frac
    for _ in range(args.warmup):
        oracle_gemm(host, frac)
    t0 = time.perf_counter()
    nbytes = 0
    for _ in range(args.steps):
        nbytes = oracle_gemm(host, frac)
    dt = (time.perf_counter() - t0) / args.steps
    value = nbytes / dt / 1e9
    cb = {"value": round(value, 4), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
          "sample": "per step: %.4g of every weight matrix's output rows of the cfg1 W4A16 layer set "
                    "(all 16 rows, full K), double precision" % frac}
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": "cfg1 W4A16 layer set at M=16 (CPU oracle sample)", "M": M_VERIFY,
                       "bytes_per_step": nbytes, "parallelism": "host cores"},
            "cpu_baseline": cb,
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-sweep", dest="sweep", action="store_false")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-prefill", dest="prefill", action="store_false")
    ap.add_argument("--prefill-only", action="store_true", help="run only the prefill leg (profiling aid)")
    ap.add_argument("--gdn-only", action="store_true", help="run only the gated-delta state leg (profiling aid)")
    ap.add_argument("--lmhead-only", action="store_true",
                    help="run only the batched lm_head leg (8 x 16 rows, then the last row; profiling aid)")
    ap.add_argument("--ref-frac", type=float, default=1.0 / 16)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    if args.prefill_only or args.gdn_only or args.lmhead_only:
        import torch
        from speculative_decoding_verify_w4a16_gb300 import _build, w4v
        _build.build()
        w4v.load()
        w4v.init()
        dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
        if args.prefill_only:
            out, leg = {"prefill": run_prefill(dev, w4v, torch, load_peaks())}, "prefill"
        elif args.lmhead_only:
            out, leg = {"lmhead_batched": run_lmhead_batched(dev, w4v, torch, load_peaks())}, "batched lm_head"
        else:
            out, leg = {"gdn_state": run_gdn(dev, w4v, torch)}, "recurrent state"
        check_device_status(w4v, leg)
        print(json.dumps(out), flush=True)
        return
    res = run_gpu(args, rank, world)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
