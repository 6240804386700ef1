#!/usr/bin/env python
"""Benchmark of the 2-bit MoE layer (moe_w2_forward) and the NVFP4 re-quantizer.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

Default workload: decode_t1 (H=6144, I=2048, E=256, top-8, T=1, Zipf(1.1)
routing), the single-token decode step.  One step = one moe_w2_forward of one
batch: permutation, gate_up with SiLU*up, down with the weighted combine.  The
default single-GPU run also measures the other full-size workloads, decode_t32,
prefill_t8192 and requant_256, and adds one object per workload under
"configs" in the same JSON line (value, ms_per_step, roofline, e2e, cpu_baseline).

Timing: inputs are resident in HBM; every step replays a captured CUDA graph of
the forward, timed by CUDA events recorded on the launching stream around the
replay (step time, `value`).  A second timed pass over the same steps replays
graphs of moe_w2_forward_traced, whose phase events give each kernel's time (the
roofline line); its step time is reported as ms_per_step_traced.  L2 is flushed
(a 512 MiB write) before every step, outside the timed events.  Routings rotate
over a pool, so consecutive steps touch different experts.  SM clocks and
throttle reasons are sampled with nvidia-smi (by the timed GPU's PCI bus id)
from before the warm-up through the timed steps, with extra untimed replays
before the timed ones so that at least ten samples fall under load.  "e2e" times the same call with the step's inputs
copied from pinned host memory and y copied back inside the timed events.

--impl reference runs the CPU oracle (plain C, single-threaded) on a bounded
sample of the same workload on this host; it never touches the GPU.  Each
cpu_baseline also reports the OpenMP build of the same oracle on all host cores.
Multi-GPU (torchrun): independent replicas, one per GPU (the layer has no
cross-GPU step on one box); value = all ranks' tokens / slowest rank's time.
"""
from __future__ import annotations

import argparse
import ctypes
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from bit_moe_expert_w2_gb300 import inputs  # noqa: E402

METRIC = "w2 MoE layer tokens/s; plane HBM GB/s (decode), TFLOP/s (prefill) vs peak"
DEFAULT_CONFIG = "decode_t1"
EXTRA_CONFIGS = ("decode_t32", "prefill_t8192", "w4_decode_t1_e64", "w4_prefill_t8192_e64", "requant_256",
                 "requant_fp8_16", "requant_mxfp4_16")
DEFAULT_STEPS = {"decode_t1": 4000, "decode_t32": 1000, "prefill_t8192": 100, "requant_256": 10,
                 "decode_t1_e32": 4000, "prefill_t1024_e32": 400}
EXTRA_STEPS = {"decode_t32": 500, "prefill_t8192": 50, "w4_decode_t1_e64": 2000, "w4_prefill_t8192_e64": 30,
               "requant_256": 5, "requant_fp8_16": 5, "requant_mxfp4_16": 5}
POOL = 16
# every file each kernel's translation unit compiles: a capture is stale once any changed
KERNEL_SOURCES = {
    "decode_layer_kernel": ["bit_moe_expert_w2_gb300/csrc/decode.cu"],
    "decode_mma_kernel": ["bit_moe_expert_w2_gb300/csrc/decode_mma.cu"],
    "decode_stream_kernel": ["bit_moe_expert_w2_gb300/csrc/decode_stream.cu"],
    "prefill_gate_up_kernel": ["bit_moe_expert_w2_gb300/csrc/prefill.cu"],
    "requant_kernel": ["bit_moe_expert_w2_gb300/csrc/requant.cu"],
    "requant_fp8_kernel": ["bit_moe_expert_w2_gb300/csrc/requant.cu"],
}
COMMON_SOURCES = ["bit_moe_expert_w2_gb300/csrc/common.cuh", "bit_moe_expert_w2_gb300/csrc/tc.cuh", "include/moe_w2.h"]


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def sources_sha(rels) -> str:
    """One hash over the listed files (path and contents, in order)."""
    h = hashlib.sha256()
    for rel in rels:
        h.update(rel.encode() + b"\0")
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def kernel_sources(kernel: str):
    return KERNEL_SOURCES[kernel] + COMMON_SOURCES


def ncu_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, or None if
    the summary is missing or any file the kernel compiles changed since the capture."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            table = json.load(f)
    except (OSError, ValueError):
        return None
    # entries are keyed "kernel:workload" (a kernel measured on several workloads) or "kernel"
    d = table.get(f"{kernel}:{workload}") or table.get(kernel)
    if d is None:
        return None
    if d.get("workload") != workload or d.get("sources") != kernel_sources(kernel):
        return None
    if d.get("sources_sha") != sources_sha(d["sources"]):
        return None
    return d.get("traffic_bytes_per_launch")


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons of the timed GPU.

    Started before the warm-up; each sample carries the host time it arrived, so
    the summary can take the samples of a window (the timed steps, widened to the
    warm replays just before them when the timed steps alone are too short)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 100

    def __init__(self, device_id: str):
        self.device_id = device_id
        self.proc = None
        self.samples = []   # (host time, line)

    @staticmethod
    def device_id_of(torch_device) -> str:
        """nvidia-smi --id for a torch CUDA device: its PCI bus id (robust to CUDA_VISIBLE_DEVICES)."""
        import torch
        p = torch.cuda.get_device_properties(torch_device)
        try:
            return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
        except AttributeError:
            return str(torch.device(torch_device).index or 0)

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.device_id}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def wait_first(self, timeout_s: float = 5.0):
        t0 = time.time()
        while self.proc is not None and not self.samples and time.time() - t0 < timeout_s:
            time.sleep(0.01)

    def count_since(self, t0: float) -> int:
        return sum(1 for t, _ in self.samples if t >= t0)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float, warm0: float | None = None, want: int = 10):
        """Median SM clock and the throttle reasons seen in [t0, t1]; with fewer than
        `want` samples there, over [warm0, t1] (the warm replays right before)."""
        def pick(a):
            return [line for t, line in self.samples if a <= t <= t1 + self.PERIOD_MS / 1e3]
        lines, window = pick(t0), "timed steps"
        if len(lines) < want and warm0 is not None:
            lines, window = pick(warm0), "warm replays and timed steps"
        sms, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sms), "window": window, "gpu": self.device_id}


# ------------------------------------------------------------------ distributed

def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle timing

def oracle_layer_rate(lay: inputs.LayerInputs, budget_s: float, max_tokens: int | None = None):
    """Tokens/s of the oracle on whole tokens of this workload (single thread)."""
    import oracle
    oracle.lib()
    done, t0 = 0, time.perf_counter()
    T = lay.x.shape[0]
    while True:
        tok = np.array([done % T], np.int64)
        fwd = oracle.forward_tokens_w4 if "w13_e2m1" in lay.planes else oracle.forward_tokens
        fwd(lay.x, lay.ids, lay.weights, lay.planes, tokens=tok)
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_tokens is not None and done >= max_tokens):
            return done / el, done, el


def oracle_layer_rate_all_cores(lay: inputs.LayerInputs, budget_s: float):
    """Tokens/s of the OpenMP oracle on all host cores: rounds of one whole token
    per thread (the workload's tokens in turn, repeated when it has fewer tokens
    than threads), until the budget is spent."""
    import oracle
    threads = oracle.threads(parallel=True)
    T = lay.x.shape[0]
    done, t0 = 0, time.perf_counter()
    while True:
        tok = (np.arange(done, done + threads) % T).astype(np.int64)
        fwd = oracle.forward_tokens_w4 if "w13_e2m1" in lay.planes else oracle.forward_tokens
        fwd(lay.x, lay.ids, lay.weights, lay.planes, tokens=tok, parallel=True)
        done += threads
        el = time.perf_counter() - t0
        if el >= budget_s:
            return done / el, done, el, threads


def oracle_requant_rate_all_cores(gu: inputs.Nvfp4Tensors, budget_s: float):
    """Elements/s of the OpenMP oracle requant on all host cores, whole tensors in turn."""
    import oracle
    threads = oracle.threads(parallel=True)
    done_el, t0, i = 0, time.perf_counter(), 0
    n = gu.e2m1.shape[0]
    while True:
        sl = slice(i % n, i % n + 2)
        oracle.requant(gu.e2m1[sl], gu.e4m3[sl], gu.scale_2[sl], parallel=True)
        done_el += gu.e2m1[sl].size * 2
        i += 2
        el = time.perf_counter() - t0
        if el >= budget_s:
            return done_el / el, i, el, threads


def oracle_requant_fp8_rate(gu, budget_s: float, parallel: bool = False):
    """Elements/s of the oracle FP8 or MXFP4 requant on whole tensors in turn (single thread, or all threads)."""
    import oracle
    threads = oracle.threads(parallel=True) if parallel else 1
    done_el, t0, i = 0, time.perf_counter(), 0
    mx = isinstance(gu, inputs.Mxfp4Tensors)
    n = gu.e2m1.shape[0] if mx else gu.w8.shape[0]
    while True:
        sl = slice(i % n, i % n + 1)
        if mx:
            oracle.requant_mxfp4(gu.e2m1[sl], gu.scales[sl], parallel=parallel)
            done_el += gu.e2m1[sl].size * 2
        else:
            oracle.requant_fp8(gu.w8[sl], gu.scales[sl], parallel=parallel)
            done_el += gu.w8[sl].size
        i += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            return done_el / el, i, el, threads


def oracle_requant_rate(gu: inputs.Nvfp4Tensors, budget_s: float):
    """Elements/s of the oracle requant on whole tensors (single thread)."""
    import oracle
    oracle.lib()
    done_el, t0, i = 0, time.perf_counter(), 0
    while True:
        sl = slice(i % gu.e2m1.shape[0], i % gu.e2m1.shape[0] + 1)
        oracle.requant(gu.e2m1[sl], gu.e4m3[sl], gu.scale_2[sl])
        done_el += gu.e2m1[sl].size * 2
        i += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            return done_el / el, i, el


# ------------------------------------------------------------------ layer benchmark

def layer_bench(cfg: inputs.LayerConfig, steps, warmup, world, rank, local, w4: bool = False):
    """The 2-bit layer (moe_w2_forward), or with w4 the FP4 layer (moe_w4_forward)."""
    import torch
    from bit_moe_expert_w2_gb300 import moe_w2

    dev = torch.device("cuda", local)
    lay = inputs.w4_layer_inputs(cfg) if w4 else inputs.layer_inputs(cfg)
    T, H, I, E, k = cfg.tokens, cfg.hidden, cfg.inter, cfg.num_experts, cfg.top_k
    decode = T <= moe_w2.DECODE_MAX_TOKENS
    pool = POOL if decode else 2

    # step inputs: the configuration's own batch first, then fresh draws of the same recipe
    rng = np.random.default_rng(cfg.seed + 1000)
    pop = inputs.zipf_popularity(np.random.default_rng(cfg.seed + 2000), E) if cfg.routing == "zipf" else None
    batches = [(lay.x, lay.ids, lay.weights)]
    for _ in range(pool - 1):
        x = inputs.activations(rng, T, H)
        ids, w = inputs.routing(rng, cfg, popularity=pop)
        batches.append((x, ids, w))

    planes = {kk: torch.from_numpy(v).to(dev) for kk, v in lay.planes.items()}
    P = moe_w2.make_w4_planes(planes) if w4 else moe_w2.make_planes(planes)
    ws_bytes = (moe_w2.w4_workspace_size if w4 else moe_w2.workspace_size)(T, k, E, H, I)
    work = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    def to_dev(x, ids, w):
        return (torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16),
                torch.from_numpy(ids).to(dev), torch.from_numpy(w).to(dev))

    dev_batches = [to_dev(*b) for b in batches]
    ys = [torch.empty((T, H), dtype=torch.bfloat16, device=dev) for _ in range(pool)]
    # algorithmic plane bytes each step reads: every distinct expert's four sections, once
    # (FP4 layer: e2m1 and e4m3 bytes, and the three scale_2 floats)
    if w4:
        w13_b = 2 * I * (H // 2 + H // 16) + 8
        w2_b = H * (I // 2 + I // 16) + 4
    else:
        w13_b = 2 * I * (H // 4 + H // 32)
        w2_b = H * (I // 4 + I // 32)
    distinct = [len(np.unique(b[1][(b[1] >= 0) & (b[1] < E)])) for b in batches]

    L = moe_w2.load()
    f_plain = L.moe_w4_forward if w4 else L.moe_w2_forward
    f_traced = L.moe_w4_forward_traced if w4 else L.moe_w2_forward_traced
    stream = torch.cuda.Stream(device=dev)
    n_ev = 4

    def make_events():
        # torch only reports elapsed time for events it has recorded once itself;
        # the library re-records them (as graph nodes) on every replay
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
        for e in evs:
            e.record(stream)
        return evs

    def call(i, evs, s):
        x, ids, w = dev_batches[i]
        ev_ptrs = (ctypes.c_void_p * 4)(*[ctypes.c_void_p(e.cuda_event) for e in evs])
        st = f_traced(moe_w2._ptr(x), moe_w2._ptr(ids), moe_w2._ptr(w), ctypes.byref(P), T, k,
                      moe_w2._ptr(ys[i]), moe_w2._ptr(work), work.numel(), moe_w2._ptr(status),
                      ctypes.c_void_p(s.cuda_stream), ev_ptrs)
        if st != 0:
            raise moe_w2.MoeW2Error(st, "forward (traced)")

    def call_plain(i, s):
        x, ids, w = dev_batches[i]
        st = f_plain(moe_w2._ptr(x), moe_w2._ptr(ids), moe_w2._ptr(w), ctypes.byref(P), T, k,
                     moe_w2._ptr(ys[i]), moe_w2._ptr(work), work.numel(), moe_w2._ptr(status),
                     ctypes.c_void_p(s.cuda_stream))
        if st != 0:
            raise moe_w2.MoeW2Error(st, "forward")

    # two graphs per pool entry: the plain forward (timed for the step time and
    # `value`) and the traced forward with phase events (timed for the per-kernel
    # breakdown and the roofline), so the event nodes never count in the step time
    graphs, graphs_traced, events = [], [], []
    with torch.cuda.stream(stream):
        for i in range(pool):            # warm the library's one-time queries outside capture
            evs = make_events()
            call(i, evs, stream)
            call_plain(i, stream)
        torch.cuda.synchronize(dev)
        for i in range(pool):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                call_plain(i, stream)
            graphs.append(g)
            evs = make_events()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                call(i, evs, stream)
            graphs_traced.append(g)
            events.append(evs)
    torch.cuda.synchronize(dev)
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(pool)]

    def run_steps(nsteps, record):
        """Plain graphs; CUDA events on the stream around each replay (L2 flush outside)."""
        steps_total = 0.0
        per_step = []
        done = 0
        while done < nsteps:
            m = min(pool, nsteps - done)
            with torch.cuda.stream(stream):
                for j in range(m):
                    flush.zero_()
                    step_ev[j][0].record(stream)
                    graphs[(done + j) % pool].replay()
                    step_ev[j][1].record(stream)
            stream.synchronize()
            for j in range(m):
                step = step_ev[j][0].elapsed_time(step_ev[j][1])
                if record:
                    steps_total += step
                    per_step.append(((done + j) % pool, step))
            done += m
        return steps_total, per_step

    def run_traced(nsteps, eager=True):
        """Traced steps: per-phase times from the events between the kernels.  Eager
        launches (queued behind the L2 flush, so the GPU never waits on the host)
        by default; graph replays with event nodes otherwise."""
        tot = np.zeros(n_ev - 1)
        steps_total = 0.0
        done = 0
        while done < nsteps:
            m = min(pool, nsteps - done)
            with torch.cuda.stream(stream):
                for j in range(m):
                    flush.zero_()
                    if eager:
                        call((done + j) % pool, events[(done + j) % pool], stream)
                    else:
                        graphs_traced[(done + j) % pool].replay()
            stream.synchronize()
            for j in range(m):
                evs = events[(done + j) % pool]
                tot += [evs[q].elapsed_time(evs[q + 1]) for q in range(n_ev - 1)]
                steps_total += evs[0].elapsed_time(evs[n_ev - 1])
            done += m
        return steps_total, tot

    clk = ClockSampler(ClockSampler.device_id_of(dev)).start()
    clk.wait_first()
    run_steps(max(warmup, 3), False)
    run_traced(max(warmup, 3))
    # untimed replays until the clock sampler has seen the GPU under load for a while
    warm0 = time.time()
    while clk.count_since(warm0) < 10 and time.time() - warm0 < 5.0:
        run_steps(pool, False)
    barrier(world)
    torch.cuda.synchronize(dev)
    t_timed0 = time.time()
    wall0 = time.perf_counter()
    steps_ms, per_step = run_steps(steps, True)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    t_timed1 = time.time()
    traced_ms, phase_ms = run_traced(steps)
    torch.cuda.synchronize(dev)
    clk.stop()
    barrier(world)
    steps_ms_max = max_over_ranks(steps_ms, world)
    K = steps
    value = world * T * K / (steps_ms_max / 1e3)
    st_val = int(status.item())
    if st_val != 0:
        raise RuntimeError(f"device status {st_val} during the benchmark")

    pk = peaks()
    plane_bytes = sum(distinct[i] * (w13_b + w2_b) for i, _ in per_step)
    if decode:
        # context for the roofline: a plain read of the same number of bytes (a torch
        # reduction over a buffer of one step's mean plane bytes), L2 flushed and
        # timed by events around the one launch like the step; at a few tens of MB
        # the launch and the ramp of the memory system alone keep it well below peak
        nb = int(plane_bytes / steps) // 64 * 64
        rbuf = torch.ones(nb // 8, dtype=torch.int64, device=dev)
        racc = torch.empty((), dtype=torch.int64, device=dev)
        r_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(20)]
        with torch.cuda.stream(stream):
            for e0, e1 in r_ev:
                flush.zero_()
                e0.record(stream)
                torch.sum(rbuf, dim=0, out=racc)
                e1.record(stream)
        stream.synchronize()
        r_us = sorted(a.elapsed_time(b) for a, b in r_ev[3:])[len(r_ev[3:]) // 2] * 1e3
        same_size_read = {"bytes": nb, "us": round(r_us, 2), "gbs": round(nb / r_us / 1e3, 1),
                          "frac": round(nb / r_us / 1e3 / pk["hbm_gbs"], 4),
                          "how": "torch.sum over an int64 buffer of the step's plane bytes, L2 flushed, median of 17"}
        del rbuf
    res = {"ms_per_step": steps_ms / K, "ms_per_step_traced": traced_ms / K}
    if decode:
        # one kernel streams the w13 and w2 planes of every active expert; its
        # time is phase 1 (phase 2: the combine kernel, empty when the layer
        # kernel combines itself)
        kname = "decode_mma_kernel" if w4 else moe_w2.decode_kernel(T, k, H, I)
        layer_kernel_ms = phase_ms[1]
        achieved = plane_bytes / (layer_kernel_ms / 1e3) / 1e9
        res["roofline"] = {"kernel": kname, "bound": "hbm", "achieved": round(achieved, 1),
                           "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4),
                           "peak_source": pk["source"],
                           "traffic": ncu_traffic(kname, cfg.name),
                           "algorithmic_bytes_per_step": int(plane_bytes / steps),
                           "same_size_read": same_size_read}
        res["plane_gbs_step"] = round(plane_bytes / (steps_ms / 1e3) / 1e9, 1)
        res["plane_frac_step"] = round(plane_bytes / (steps_ms / 1e3) / 1e9 / pk["hbm_gbs"], 4)
    else:
        flops_gu = 2.0 * T * k * 2 * I * H
        achieved = flops_gu / (phase_ms[1] / 1e3) / 1e12 * K
        res["roofline"] = {"kernel": "prefill_gate_up_kernel", "bound": "tensor", "achieved": round(achieved, 1),
                           "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                           "frac": round(achieved / pk["bf16_tflops"], 4), "peak_source": pk["source"],
                           "traffic": ncu_traffic("prefill_gate_up_kernel", cfg.name)}
        res["layer_tflops"] = round(6.0 * T * k * H * I * K / (steps_ms / 1e3) / 1e12, 1)
    if decode:
        res["phase_ms_per_step"] = {"permute": round(phase_ms[0] / K, 5), "layer": round(phase_ms[1] / K, 5),
                                    "combine": round(phase_ms[2] / K, 5)}
    else:
        res["phase_ms_per_step"] = {"permute_gather": round(phase_ms[0] / K, 5), "gate_up": round(phase_ms[1] / K, 5),
                                    "down_combine": round(phase_ms[2] / K, 5)}
    res["distinct_experts_per_step"] = round(float(np.mean([distinct[i] for i, _ in per_step])), 2)
    res["clocks"] = clk.summary(t_timed0, t_timed1, warm0)
    res["wall_s"] = round(wall, 3)
    # decode: permute (+ x as T16 bf16 or e2m1 digit rows), the layer kernel (gate_up, down), and the
    # combine kernel after the block-scaled one;
    # prefill: permute, gather, gate_up, down, combine
    block_scaled = decode and not w4 and moe_w2.decode_kernel(T, k, H, I) == "decode_layer_kernel"
    res["kernels_per_step"] = (3 if block_scaled else 2) if decode else 5
    # arithmetic of the layer's contractions: the block-scaled decode kernel multiplies e2m1
    # weights by eight e2m1 digit rows per activation row under UE8M0 block scales; the others
    # bf16 (the FP4 layer's weights are the exact bf16 products e2m1 x e4m3)
    res["dtype"] = ("e2m1 x e2m1 digits block-scaled, fp32 accumulation" if block_scaled
                    else "bf16 (exact e2m1 x e4m3 weights), fp32 accumulation" if w4 else "bf16, fp32 accumulation")

    # end to end: pinned host inputs -> device -> forward -> y back to pinned host.  A step's
    # x, ids and weights sit back to back in one pinned buffer, so they cross in one copy
    nx, ni = T * H * 2, T * k * 4
    def packed(b):
        buf = torch.empty(nx + 2 * ni, dtype=torch.uint8).pin_memory()
        buf[:nx].copy_(torch.from_numpy(b[0].view(np.uint8).reshape(-1)))
        buf[nx:nx + ni].copy_(torch.from_numpy(b[1].view(np.uint8).reshape(-1)))
        buf[nx + ni:].copy_(torch.from_numpy(b[2].view(np.uint8).reshape(-1)))
        return buf
    hin = [packed(b) for b in batches]
    hy = [torch.empty((T, H), dtype=torch.int16).pin_memory() for _ in range(pool)]
    din = torch.empty(nx + 2 * ni, dtype=torch.uint8, device=dev)
    dx = din[:nx].view(torch.int16).view(T, H)
    did = din[nx:nx + ni].view(torch.int32).view(T, k)
    dw = din[nx + ni:].view(torch.float32).view(T, k)
    dy = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    e_start = [torch.cuda.Event(enable_timing=True) for _ in range(pool)]
    e_end = [torch.cuda.Event(enable_timing=True) for _ in range(pool)]

    def e2e_step(i):
        e_start[i].record(stream)
        din.copy_(hin[i], non_blocking=True)
        st = f_plain(moe_w2._ptr(dx), moe_w2._ptr(did), moe_w2._ptr(dw), ctypes.byref(P), T, k,
                     moe_w2._ptr(dy), moe_w2._ptr(work), work.numel(), moe_w2._ptr(status),
                     ctypes.c_void_p(stream.cuda_stream))
        if st != 0:
            raise moe_w2.MoeW2Error(st, "forward")
        hy[i].copy_(dy.view(torch.int16), non_blocking=True)
        e_end[i].record(stream)

    with torch.cuda.stream(stream):
        for i in range(pool):
            e2e_step(i)
    stream.synchronize()
    e2e_ms, done = 0.0, 0
    barrier(world)
    while done < steps:
        m = min(pool, steps - done)
        with torch.cuda.stream(stream):
            for j in range(m):
                flush.zero_()
                e2e_step(j)
        stream.synchronize()
        e2e_ms += sum(e_start[j].elapsed_time(e_end[j]) for j in range(m))
        done += m
    e2e_ms = max_over_ranks(e2e_ms, world)
    bytes_in = batches[0][0].nbytes + batches[0][1].nbytes + batches[0][2].nbytes
    res["e2e"] = {"value": round(world * T * steps / (e2e_ms / 1e3), 2), "unit": "tokens/s",
                  "h2d_bytes_per_step": int(bytes_in), "d2h_bytes_per_step": int(T * H * 2)}
    res["gpu_launches"] = res["kernels_per_step"] * steps
    res["value"] = value
    return res, lay


def requant_bench(name, steps, warmup, world, rank, local):
    import torch
    from bit_moe_expert_w2_gb300 import moe_w2
    dev = torch.device("cuda", local)
    gu, dn = inputs.requant_inputs(experts=inputs.REQUANT_CASES[name])
    dgu = [torch.from_numpy(a).to(dev) for a in (gu.e2m1, gu.e4m3, gu.scale_2)]
    ddn = [torch.from_numpy(a).to(dev) for a in (dn.e2m1, dn.e4m3, dn.scale_2)]
    cgu = torch.empty((gu.e2m1.shape[0], gu.e2m1.shape[1], gu.e2m1.shape[2] // 2), dtype=torch.uint8, device=dev)
    sgu = torch.empty((gu.e2m1.shape[0], gu.e2m1.shape[1], gu.e2m1.shape[2] // 16), dtype=torch.uint8, device=dev)
    cdn = torch.empty((dn.e2m1.shape[0], dn.e2m1.shape[1], dn.e2m1.shape[2] // 2), dtype=torch.uint8, device=dev)
    sdn = torch.empty((dn.e2m1.shape[0], dn.e2m1.shape[1], dn.e2m1.shape[2] // 16), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]

    def step(e0=None, e1=None):
        if e0 is not None:
            e0.record(stream)
        moe_w2.requant(*dgu, codes=cgu, ue8m0=sgu, status=status, stream=stream)
        moe_w2.requant(*ddn, codes=cdn, ue8m0=sdn, status=status, stream=stream)
        if e1 is not None:
            e1.record(stream)

    clk = ClockSampler(ClockSampler.device_id_of(dev)).start()
    clk.wait_first()
    with torch.cuda.stream(stream):
        for _ in range(max(warmup, 3)):
            step()
    stream.synchronize()
    warm0 = time.time()
    while clk.count_since(warm0) < 10 and time.time() - warm0 < 5.0:
        with torch.cuda.stream(stream):
            step()
        stream.synchronize()
    barrier(world)
    t_timed0 = time.time()
    with torch.cuda.stream(stream):
        for e0, e1 in evs:
            flush.zero_()
            step(e0, e1)
    stream.synchronize()
    t_timed1 = time.time()
    clk.stop()
    ms = sum(a.elapsed_time(b) for a, b in evs)
    ms = max_over_ranks(ms, world)
    elems = gu.e2m1.size * 2 + dn.e2m1.size * 2
    moved = sum(a.nbytes for a in (gu.e2m1, gu.e4m3, dn.e2m1, dn.e4m3)) + elems // 4 + elems // 32
    pk = peaks()
    gbs = moved * steps / (ms / 1e3) / 1e9
    res = {"ms_per_step": ms / steps, "value": world * elems * steps / (ms / 1e3),
           "roofline": {"kernel": "requant_kernel", "bound": "hbm", "achieved": round(gbs, 1),
                        "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(gbs / pk["hbm_gbs"], 4),
                        "peak_source": pk["source"], "traffic": ncu_traffic("requant_kernel", name),
                        "algorithmic_bytes_per_step": int(moved)},
           "clocks": clk.summary(t_timed0, t_timed1, warm0), "gpu_launches": 2 * steps, "dtype": "int64 (exact)"}

    # end to end: the NVFP4 tensors from pinned host memory, requant, planes back to pinned host memory
    hin = [torch.from_numpy(a).pin_memory() for a in (gu.e2m1, gu.e4m3, gu.scale_2, dn.e2m1, dn.e4m3, dn.scale_2)]
    hout = [torch.empty(t.shape, dtype=torch.uint8).pin_memory() for t in (cgu, sgu, cdn, sdn)]
    e_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for e0, e1 in e_evs:
            flush.zero_()
            e0.record(stream)
            for d, h in zip(dgu + ddn, hin):
                d.copy_(h, non_blocking=True)
            moe_w2.requant(*dgu, codes=cgu, ue8m0=sgu, status=status, stream=stream)
            moe_w2.requant(*ddn, codes=cdn, ue8m0=sdn, status=status, stream=stream)
            for h, d in zip(hout, (cgu, sgu, cdn, sdn)):
                h.copy_(d, non_blocking=True)
            e1.record(stream)
    stream.synchronize()
    e2e_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in e_evs), world)
    res["e2e"] = {"value": round(world * elems * steps / (e2e_ms / 1e3), 2), "unit": "elements/s",
                  "h2d_bytes_per_step": int(sum(h.nbytes for h in hin)),
                  "d2h_bytes_per_step": int(sum(h.nbytes for h in hout))}
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} during the requant benchmark")
    return res, gu


def loader_bench(name, steps, warmup, world, rank, local):
    """The FP8 block-128 and MXFP4 loaders on their 16-expert workloads."""
    import torch
    from bit_moe_expert_w2_gb300 import moe_w2
    dev = torch.device("cuda", local)
    fp8 = name in inputs.REQUANT_FP8_CASES
    if fp8:
        gu, dn = inputs.requant_fp8_inputs(experts=inputs.REQUANT_FP8_CASES[name])
        arrays = [(t.w8, t.scales) for t in (gu, dn)]
        K_of = lambda a: a.shape[2]
        call, kernel = moe_w2.requant_fp8, "requant_fp8_kernel"
    else:
        gu, dn = inputs.requant_mxfp4_inputs(experts=inputs.REQUANT_MXFP4_CASES[name])
        arrays = [(t.e2m1, t.scales) for t in (gu, dn)]
        K_of = lambda a: a.shape[2] * 2
        call, kernel = moe_w2.requant_mxfp4, "requant_kernel"
    dt = [(torch.from_numpy(a).to(dev), torch.from_numpy(b).to(dev)) for a, b in arrays]
    outs = [(torch.empty((a.shape[0], a.shape[1], K_of(a) // 4), dtype=torch.uint8, device=dev),
             torch.empty((a.shape[0], a.shape[1], K_of(a) // 32), dtype=torch.uint8, device=dev))
            for a, _ in arrays]
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step():
        for (w, sc), (c, u) in zip(dt, outs):
            call(w, sc, codes=c, ue8m0=u, status=status, stream=stream)

    clk = ClockSampler(ClockSampler.device_id_of(dev)).start()
    clk.wait_first()
    with torch.cuda.stream(stream):
        for _ in range(max(warmup, 3)):
            step()
    stream.synchronize()
    warm0 = time.time()
    while clk.count_since(warm0) < 10 and time.time() - warm0 < 5.0:
        with torch.cuda.stream(stream):
            step()
        stream.synchronize()
    barrier(world)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    t_timed0 = time.time()
    with torch.cuda.stream(stream):
        for e0, e1 in evs:
            flush.zero_()
            e0.record(stream)
            step()
            e1.record(stream)
    stream.synchronize()
    t_timed1 = time.time()
    clk.stop()
    ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in evs), world)
    elems = sum(a.shape[0] * a.shape[1] * K_of(a) for a, _ in arrays)
    moved = sum(a.nbytes + b.nbytes for a, b in arrays) + elems // 4 + elems // 32
    pk = peaks()
    gbs = moved * steps / (ms / 1e3) / 1e9
    res = {"ms_per_step": ms / steps, "value": world * elems * steps / (ms / 1e3), "unit": "elements/s",
           "roofline": {"kernel": kernel, "bound": "hbm", "achieved": round(gbs, 1),
                        "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(gbs / pk["hbm_gbs"], 4),
                        "peak_source": pk["source"], "traffic": ncu_traffic(kernel, name),
                        "algorithmic_bytes_per_step": int(moved)},
           "clocks": clk.summary(t_timed0, t_timed1, warm0), "gpu_launches": 2 * steps, "dtype": "int64 (exact)"}
    # end to end: the input tensors from pinned host memory, requant, planes back to pinned host memory
    hin = [(torch.from_numpy(a).pin_memory(), torch.from_numpy(b).pin_memory()) for a, b in arrays]
    hout = [(torch.empty(c.shape, dtype=torch.uint8).pin_memory(), torch.empty(u.shape, dtype=torch.uint8).pin_memory())
            for c, u in outs]
    e_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for e0, e1 in e_evs:
            flush.zero_()
            e0.record(stream)
            for (w, sc), (hw, hs) in zip(dt, hin):
                w.copy_(hw, non_blocking=True)
                sc.copy_(hs, non_blocking=True)
            step()
            for (c, u), (hc, hu) in zip(outs, hout):
                hc.copy_(c, non_blocking=True)
                hu.copy_(u, non_blocking=True)
            e1.record(stream)
    stream.synchronize()
    e2e_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in e_evs), world)
    res["e2e"] = {"value": round(world * elems * steps / (e2e_ms / 1e3), 2), "unit": "elements/s",
                  "h2d_bytes_per_step": int(sum(a.nbytes + b.nbytes for a, b in hin)),
                  "d2h_bytes_per_step": int(sum(a.nbytes + b.nbytes for a, b in hout))}
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} during the {name} benchmark")
    return res, gu


def cpu_baseline(name, data, budget_s):
    """The oracle on this host: one core (the reported value) and all cores."""
    if name in inputs.REQUANT_FP8_CASES or name in inputs.REQUANT_MXFP4_CASES:
        v, n, el, _ = oracle_requant_fp8_rate(data, budget_s)
        va, na, ela, thr = oracle_requant_fp8_rate(data, budget_s / 2, parallel=True)
        return {"value": round(v, 1), "unit": "elements/s", "cores": 1, "kind": "oracle",
                "sample": f"{n} whole tensors of {name} in {el:.1f} s",
                "all_cores": {"value": round(va, 1), "cores": thr,
                              "sample": f"{na} whole tensors in {ela:.1f} s (OpenMP build)"}}
    if name in inputs.REQUANT_CASES:
        v, n, el = oracle_requant_rate(data, budget_s)
        va, na, ela, thr = oracle_requant_rate_all_cores(data, budget_s / 2)
        return {"value": round(v, 1), "unit": "elements/s", "cores": 1, "kind": "oracle",
                "sample": f"{n} whole gate/up tensors of {name} in {el:.1f} s",
                "all_cores": {"value": round(va, 1), "cores": thr,
                              "sample": f"{na} whole gate/up tensors in {ela:.1f} s (OpenMP build)"}}
    v, n, el = oracle_layer_rate(data, budget_s)
    va, na, ela, thr = oracle_layer_rate_all_cores(data, budget_s / 2)
    return {"value": round(v, 4), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} whole tokens of {name} in {el:.1f} s",
            "all_cores": {"value": round(va, 4), "cores": thr,
                          "sample": f"{na} whole tokens in {ela:.1f} s (OpenMP build, one token per thread)"}}


def run_config(name, steps, warmup, world, rank, local):
    """(result dict, oracle input) of one workload."""
    if name in inputs.REQUANT_FP8_CASES or name in inputs.REQUANT_MXFP4_CASES:
        return loader_bench(name, steps, warmup, world, rank, local)
    if name in inputs.REQUANT_CASES:
        res, data = requant_bench(name, steps, warmup, world, rank, local)
        res["unit"] = "elements/s"
    elif name in inputs.W4_CONFIGS:
        res, data = layer_bench(inputs.W4_CONFIGS[name], steps, warmup, world, rank, local, w4=True)
        res["unit"] = "tokens/s"
    else:
        res, data = layer_bench(inputs.CONFIGS[name], steps, warmup, world, rank, local)
        res["unit"] = "tokens/s"
    return res, data


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=None,
                    choices=[*inputs.CONFIGS, *inputs.W4_CONFIGS, *inputs.REQUANT_CASES, *inputs.REQUANT_FP8_CASES,
                             *inputs.REQUANT_MXFP4_CASES],
                    help=f"one workload only (default: {DEFAULT_CONFIG}, plus {', '.join(EXTRA_CONFIGS)} on one GPU)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of single-core oracle work per workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-configs", action="store_true", help="only the headline workload")
    args = ap.parse_args()
    headline = args.config or DEFAULT_CONFIG
    if args.steps is None:
        args.steps = DEFAULT_STEPS.get(headline, 10)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    cores = len(os.sched_getaffinity(0))

    if args.impl == "reference":
        if rank != 0:
            return
        args.config = headline
        return reference_arm(args, cores)

    world, rank, local = dist_setup(args)
    res, data = run_config(headline, args.steps, args.warmup, world, rank, local)
    extras = {}
    if args.config is None and world == 1 and not args.no_extra_configs:
        for name in EXTRA_CONFIGS:
            extras[name] = run_config(name, EXTRA_STEPS[name], args.warmup, world, rank, local)
    if rank != 0:
        return
    line = {"metric": METRIC, "value": round(res.pop("value"), 3), "unit": res.pop("unit"), "n_gpus": world,
            "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(res.pop("ms_per_step"), 6),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": res.pop("dtype", "bf16"),
            "data": "synthetic (seeded; shapes of the pages' models)",
            "config": {"workload": workload_name(headline), "l2": "flushed before every step (512 MiB write, untimed)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}}
    line.update(res)
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(headline, data, args.cpu_budget)
    if extras:
        line["configs"] = {}
        for name, (r, d) in extras.items():
            obj = {"workload": workload_name(name), "value": round(r.pop("value"), 3), "unit": r.pop("unit"),
                   "steps": EXTRA_STEPS[name], "ms_per_step": round(r.pop("ms_per_step"), 6)}
            obj.update(r)
            if not args.no_cpu_baseline:
                obj["cpu_baseline"] = cpu_baseline(name, d, args.cpu_budget)
            line["configs"][name] = obj
    print(json.dumps(line), flush=True)


def workload_name(config: str) -> str:
    """The workload string of a config, the same on both arms."""
    if config in inputs.REQUANT_FP8_CASES:
        r = inputs.REQUANT
        n = inputs.REQUANT_FP8_CASES[config]
        return (f"{config}: {n} experts FP8 (e4m3, f32 128x128 block scales) gate/up 2x[{r.inter}x{r.hidden}] + "
                f"down [{r.hidden}x{r.inter}] -> 2-bit planes")
    if config in inputs.REQUANT_MXFP4_CASES:
        r = inputs.REQUANT
        n = inputs.REQUANT_MXFP4_CASES[config]
        return (f"{config}: {n} experts MXFP4 (e2m1, UE8M0 block-32 scales) gate/up 2x[{r.inter}x{r.hidden}] + "
                f"down [{r.hidden}x{r.inter}] -> 2-bit planes")
    if config in inputs.REQUANT_CASES:
        r = inputs.REQUANT
        n = inputs.REQUANT_CASES[config] or r.num_experts
        return (f"{config}: {n} experts NVFP4 gate/up 2x[{r.inter}x{r.hidden}] + down [{r.hidden}x{r.inter}]"
                " -> 2-bit planes")
    if config in inputs.W4_CONFIGS:
        cfg = inputs.W4_CONFIGS[config]
        return (f"{cfg.name}: FP4 layer (NVFP4 experts) H={cfg.hidden} I={cfg.inter} E={cfg.num_experts} "
                f"top-{cfg.top_k} T={cfg.tokens} routing={cfg.routing}")
    cfg = inputs.CONFIGS[config]
    return (f"{cfg.name}: H={cfg.hidden} I={cfg.inter} E={cfg.num_experts} top-{cfg.top_k} "
            f"T={cfg.tokens} routing={cfg.routing}")


def reference_arm(args, cores):
    """The oracle timed on this host's cores on a bounded sample of the workload."""
    budget = 90.0
    if args.config in inputs.REQUANT_FP8_CASES or args.config in inputs.REQUANT_MXFP4_CASES:
        fp8 = args.config in inputs.REQUANT_FP8_CASES
        gu, _ = (inputs.requant_fp8_inputs if fp8 else inputs.requant_mxfp4_inputs)(experts=2)
        v, n, el, _ = oracle_requant_fp8_rate(gu, budget / 3)
        unit, sample = "elements/s", f"{n} whole tensors of {args.config} in {el:.1f} s"
        steps = n
    elif args.config in inputs.REQUANT_CASES:
        gu, _ = inputs.requant_inputs(experts=4)
        v, n, el = oracle_requant_rate(gu, budget / 3)
        unit, sample = "elements/s", f"{n} whole gate/up tensors of {args.config} in {el:.1f} s"
        steps = n
    else:
        if args.config in inputs.W4_CONFIGS:
            lay = inputs.w4_layer_inputs(inputs.W4_CONFIGS[args.config])
        else:
            lay = inputs.layer_inputs(inputs.CONFIGS[args.config])
        # warm-up tokens, then timed tokens until the step count or the budget is reached
        oracle_layer_rate(lay, float("inf"), max_tokens=max(args.warmup, 3))
        v, n, el = oracle_layer_rate(lay, budget, max_tokens=args.steps)
        unit, sample = "tokens/s", f"{n} whole tokens of {args.config} in {el:.1f} s"
        steps = n
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": unit, "n_gpus": 0,
            "steps": steps, "warmup": max(args.warmup, 3), "ms_per_step": round(el / max(steps, 1) * 1e3, 3),
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": workload_name(args.config), "sample": sample},
            "cpu_baseline": {"value": round(v, 4), "unit": unit, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 4), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "host_cores_available": cores}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
