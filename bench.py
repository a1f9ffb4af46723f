#!/usr/bin/env python3
"""Benchmark of the RMSNorm + RoPE hot path on GB300; prints ONE JSON line (rank 0).

Workload (one "step"), Llama-3.2-1B-shaped prefill of 4096 tokens, bf16 storage:
  * RMSNorm  x[4096, 2048], w[2048], eps 1e-5
  * RoPE     Q[1, 4096, 32, 64] and K[1, 4096, 8, 64] rotated by one camp_rope_qk launch
             with shared fp32 sin/cos [4096, 32] (theta 500000)
76,550,144 algorithmic bytes per step (every input read once, every output written once,
the weight and the tables included).

Timing. Inputs are drawn on the device before timing. Each step uses one of R input sets
(R * step bytes > 4 x L2), so nothing a step reads is still in L2 from its last use. The
timed region runs exactly K steps as blocks of up to 1024 steps: per block, one CUDA graph
with an event node, the block's M back-to-back RMSNorm launches (input sets 0, 1, ... mod
R), its M Q+K RoPE launches and a last event node (the two operators of a step are
independent, so a block runs all of its steps' work); the event between the two runs sits
on a side branch of the graph, so that it adds no dependency between the kernels. The event
nodes give every kernel's time without events between individual launches (an event pair
around a 5 us kernel adds several microseconds). The region is timed again and again, with L2 flushed
by a read of twice its size before each repeat, for at least --repeats repeats and about --min-seconds of GPU time,
with a barrier and a device synchronize before and after; ``value`` is the step bytes x K x
ranks / the slowest rank's median region time, and a kernel's launch duration its summed
time in the median repeat / K. nvidia-smi samples the SM clock and the throttle reasons
during the repeats.

``e2e`` is the same metric through the C ABI with host buffers: every step copies its
inputs (one packed slab) from pinned host memory, runs the two kernels and copies the
outputs (one packed slab) back, double-buffered on three streams (``e2e.serial``: the same
on one stream).

``large_configs`` and ``sweep`` time each operator alone at the large shapes and at every
shape of the token x hidden / heads x head_dim sweep, as graphs of back-to-back launches
over rotating input sets (GB/s, fraction of the peak, rows/s).

``cpu_baseline`` times the fp64 oracle (test infrastructure, as it stands) on the host
cores on whole steps of the same workload, and on a bounded sample of each RMSNorm and
RoPE configuration. ``--impl reference`` prints the reference arm's line instead: that
oracle, timed on a bounded sample of the workload per step.

Multi-GPU (under torchrun): every rank runs an independent replica of the workload (the
rows are independent; there is no exchange step), so scaling is weak and ``value`` sums
over ranks.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from block_memory_bound_gb300 import camp, inputs, ledger  # noqa: E402

METRIC = "achieved HBM GB/s and % of GB300 peak for RMSNorm/RoPE (bf16, 4096×2048)"
UNIT = "GB/s"

TOKENS, HIDDEN, HQ, HK, HEAD_DIM = 4096, 2048, 32, 8, 64
EPS = 1e-5
THETA = 500000.0

BYTES_RMS = ledger.rmsnorm_bytes(TOKENS, HIDDEN, "bf16")
BYTES_RQK = ledger.rope_qk_bytes(1, TOKENS, HQ, HK, HEAD_DIM, "bf16")
STEP_BYTES = BYTES_RMS + BYTES_RQK
KERNELS = ("rmsnorm", "rope_qk")
KERNEL_BYTES = {"rmsnorm": BYTES_RMS, "rope_qk": BYTES_RQK}

WORKLOAD = ("llama3.2-1b prefill 4096 tokens: rmsnorm x[4096,2048] + rope of Q[1,4096,32,64] "
            "and K[1,4096,8,64] in one launch, bf16, shared fp32 tables [4096,32], "
            "theta 500000")

FALLBACK_HBM_GBS = 6800.0

# How the timed region keeps HBM cold; one statement for both arms so their configs match.
L2_POLICY = ("inputs larger than L2: rotating input sets of more than 4 x L2 in total, "
             "and between timed repeats a read of a buffer of 2 x L2, which evicts what the "
             "last repeat left in L2")
# Both arms print this config: N independent replicas of the workload (one per rank).
STEP_CONFIG = {"workload": WORKLOAD, "parallelism": "replicas", "step_bytes": STEP_BYTES,
               "l2": L2_POLICY}

# Where the per-kernel, large-shape, sweep and calibration figures are written (the JSON
# line on stdout stays short).
DETAIL_PATH = os.path.join("gpurun_out", "bench_detail.json")
LINE_LIMIT = 2048   # bytes of the final stdout line


# ------------------------------------------------------------------ helpers

def log(*a):
    print(*a, file=sys.stderr, flush=True)


def load_peak() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# The device sources each recorded kernel is built from (profiles/traffic.json): a
# recorded DRAM figure is reported only while these files are unchanged.
KERNEL_SOURCES = {
    "rope_tiled": ("rope.cu", "common.cuh", "kernels.h"),
    "rmsnorm_rows": ("rmsnorm.cu", "rmsnorm_kernels.cuh", "common.cuh", "kernels.h"),
}


def source_digest(names=None) -> str:
    """Digest of device code: the named files of csrc/, or every kernel source and header
    (camp_abi.cu, host-only planning and argument checks, left out: it cannot change what a
    kernel variant moves)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_memory_bound_gb300", "csrc")
    files = sorted(names) if names else sorted(
        n for n in os.listdir(csrc) if n.endswith((".cu", ".cuh", ".h")) and n != "camp_abi.cu")
    for name in files:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def recorded_traffic(kernel_name: str):
    """DRAM bytes per launch from the committed ncu summary, if its kernel's sources are
    the ones it was recorded from."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get("kernels", {}).get(kernel_name)
    if entry is None:
        return None
    family = kernel_name.split("<")[0]
    if entry.get("source_sha256") != source_digest(KERNEL_SOURCES.get(family)):
        return None
    return entry.get("dram_bytes_per_launch")


def plan_name(kind: str, p: camp.Plan, dt: str = "bf16") -> str:
    if p.kernel in (camp.KERNEL_RMSNORM_SPREAD, camp.KERNEL_LAYERNORM_SPREAD):
        return f"{kind}_spread<{dt},cluster{p.cluster},chunk{p.group}vec,stages{p.per_thread}>"
    if kind == "layernorm":
        if p.kernel == camp.KERNEL_LAYERNORM_STAGED:
            return (f"layernorm_staged<{dt},cluster{p.cluster},chunk{p.group}vec,"
                    f"stages{p.per_thread}>")
        if p.kernel == camp.KERNEL_LAYERNORM_WIDE:
            return f"layernorm_wide<{dt},vec{p.vec_bytes}>"
        return f"layernorm_rows<{dt},vec{p.vec_bytes},group{p.group},nv{p.per_thread}>"
    if kind == "rmsnorm":
        if p.kernel == camp.KERNEL_RMSNORM_STAGED:
            return (f"rmsnorm_staged<{dt},cluster{p.cluster},chunk{p.group}vec,"
                    f"stages{p.per_thread}>")
        k = {camp.KERNEL_RMSNORM_ROWS: "rmsnorm_rows", camp.KERNEL_RMSNORM_CLUSTER: "rmsnorm_cluster",
             camp.KERNEL_RMSNORM_WIDE: "rmsnorm_wide"}.get(p.kernel, "rmsnorm")
        extra = f",cluster{p.cluster}" if p.kernel == camp.KERNEL_RMSNORM_CLUSTER else ""
        return f"{k}<{dt},vec{p.vec_bytes},group{p.group},nv{p.per_thread}{extra}>"
    k = {camp.KERNEL_ROPE: "rope_tiled", camp.KERNEL_ROPE_FLAT: "rope_flat",
         camp.KERNEL_ROPE_SPLIT: "rope_split"}.get(p.kernel, "rope")
    return f"{k}<{dt},vec{p.vec_bytes},hpt{p.group}>"


class ClockSampler:
    """nvidia-smi samples (every 100 ms) of SM clock, power and throttle reasons."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self, t0: float, t1: float) -> dict:
        import datetime
        sm, mx, pw, reasons, n = [], [], [], set(), 0
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            f = [c.strip() for c in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            if not (t0 <= ts <= t1):
                continue
            n += 1
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
                pw.append(float(f[3]))
            except ValueError:
                pass
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": sorted(reasons), "samples": n}


# ------------------------------------------------------------------ ranks

def ranks_max(values: list[float], dist, device: str = "cuda") -> list[float]:
    """Element-wise maximum of `values` over all ranks (the slowest rank's times); the
    values themselves when there is no process group."""
    if dist is None:
        return list(values)
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_value(step_bytes: int, steps: int, world: int, seconds: float) -> float:
    """Whole-job GB/s: every rank runs its own replica of `steps` steps of `step_bytes`
    (weak scaling), and the job takes the slowest rank's `seconds`."""
    return step_bytes * steps * world / seconds / 1e9


# ------------------------------------------------------------------ the workload

class InputSet:
    """One set of step inputs and outputs on the device (raw pointers cached)."""

    def __init__(self, seed: int, device):
        self.x, self.w = inputs.rmsnorm_inputs(TOKENS, HIDDEN, "bf16", seed=seed, device=device)
        self.y = torch.empty_like(self.x)
        self.q, self.sq, self.cq = inputs.rope_inputs(1, TOKENS, HQ, HEAD_DIM, "bf16", seed=seed,
                                                      theta=THETA, device=device)
        self.k, _, _ = inputs.rope_inputs(1, TOKENS, HK, HEAD_DIM, "bf16", seed=seed + 500,
                                          theta=THETA, device=device)
        self.yq = torch.empty_like(self.q)
        self.yk = torch.empty_like(self.k)
        self.p = {n: t.data_ptr() for n, t in vars(self).items() if isinstance(t, torch.Tensor)}

    def inputs_(self):
        return (self.x, self.w, self.q, self.k, self.sq, self.cq)

    def outputs_(self):
        return (self.y, self.yq, self.yk)


def launch(kind: str, s: InputSet, stream: int) -> None:
    p = s.p
    if kind == "rmsnorm":
        camp.camp_rmsnorm(p["x"], p["w"], p["y"], TOKENS, HIDDEN, EPS, camp.BF16, stream)
    else:
        camp.camp_rope_qk(p["q"], p["k"], p["sq"], p["cq"], p["yq"], p["yk"], 1, TOKENS, HQ, HK,
                          HEAD_DIM, camp.BF16, stream)


def launch_step(s: InputSet, stream: int) -> None:
    for kind in KERNELS:
        launch(kind, s, stream)


def copy_calibration(sets, M: int, blocks: int, peak: float) -> dict:
    """The floor of this harness: per operator, a plain device-to-device copy of the bytes
    the operator reads (its x, or Q and K as one flat buffer) into a buffer of the same
    size, on the same rotating input sets, as CUDA graphs of M back-to-back copies timed
    with events exactly like the kernels. A copy moves its bytes twice (read + write), as
    the operators do; the weight and the tables are left out (under 3% of either)."""
    out = {}
    R = len(sets)
    for kind in KERNELS:
        if kind == "rmsnorm":
            pairs = [(s.x, torch.empty_like(s.x)) for s in sets]
        else:
            n = (sets[0].q.numel() + sets[0].k.numel()) * sets[0].q.element_size()
            pairs = [(torch.empty(n, dtype=torch.uint8, device="cuda"),
                      torch.empty(n, dtype=torch.uint8, device="cuda")) for _ in sets]
            for src, _ in pairs:
                src.random_(0, 256)
        moved = 2 * pairs[0][0].numel() * pairs[0][0].element_size()
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        with torch.cuda.graph(g, stream=cap):
            for i in range(M):
                src, dst = pairs[i % R]
                dst.copy_(src)
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(blocks):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) * 1e-3 / (blocks * M)
        out[kind] = {"bytes_moved": moved, "us": t * 1e6, "GB/s": moved / t / 1e9,
                     "frac": moved / t / 1e9 / peak}
        del g, pairs
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------ CPU legs (oracle)

def _host_step_inputs(s: InputSet) -> dict:
    return {
        "x": inputs.to_numpy(s.x), "w": inputs.to_numpy(s.w),
        "q": inputs.to_numpy(s.q), "sq": s.sq.cpu().numpy(), "cq": s.cq.cpu().numpy(),
        "k": inputs.to_numpy(s.k),
    }


def _oracle_fraction(h: dict, frac: float, lib) -> int:
    """Run the oracle on the first `frac` of every operator's rows; return bytes covered."""
    import oracle
    rows = max(1, int(round(TOKENS * frac)))
    eps32 = float(__import__("numpy").float32(EPS))
    oracle.rmsnorm(h["x"][:rows], h["w"], eps32, "bf16", lib=lib)
    oracle.rope(h["q"][:, :rows], h["sq"][:rows], h["cq"][:rows], "bf16", lib=lib)
    oracle.rope(h["k"][:, :rows], h["sq"][:rows], h["cq"][:rows], "bf16", lib=lib)
    return ledger.rmsnorm_bytes(rows, HIDDEN) + ledger.rope_qk_bytes(1, rows, HQ, HK, HEAD_DIM)


def cpu_baseline(h: dict, seconds: float) -> dict:
    import oracle
    lib = oracle.load()
    cores = oracle.threads_available(lib)
    _oracle_fraction(h, 1.0, lib)          # warm
    n, nbytes = 0, 0
    t0 = time.perf_counter()
    while True:
        nbytes += _oracle_fraction(h, 1.0, lib)
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": nbytes / dt / 1e9, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} whole steps of the workload (fp64 oracle, {cores} threads, "
                      f"{dt:.1f} s)",
            "rmsnorm_f32_64x2048_1_thread": _oracle_small_case(lib)}


def _oracle_small_case(lib) -> dict:
    """The oracle on RMSNorm fp32 x[64, 2048] (the small configuration) on one thread: the
    median of 50 calls."""
    import oracle
    x, w = inputs.rmsnorm_inputs(64, 2048, "f32", seed=0)
    xs, ws = inputs.to_numpy(x), inputs.to_numpy(w)
    eps32 = float(__import__("numpy").float32(EPS))
    ts = []
    for _ in range(51):
        t0 = time.perf_counter()
        oracle.rmsnorm(xs, ws, eps32, "f32", nthreads=1, lib=lib)
        ts.append(time.perf_counter() - t0)
    t = statistics.median(ts[1:])
    nbytes = ledger.rmsnorm_bytes(64, 2048, "f32")
    return {"us": t * 1e6, "GB/s": nbytes / t / 1e9, "threads": 1}


# ------------------------------------------------------------------ reference arm

def run_reference(args) -> None:
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np
    import oracle
    lib = oracle.load()
    cores = oracle.threads_available(lib)
    s = InputSet(0, "cpu")
    h = _host_step_inputs(s)
    # Size the per-step sample so that warm-up + steps take about args.ref_seconds.
    t0 = time.perf_counter()
    _oracle_fraction(h, 1.0 / 64, lib)
    t_full = (time.perf_counter() - t0) * 64
    frac = min(1.0, args.ref_seconds / max(1, args.steps + args.warmup) / max(t_full, 1e-9))
    frac = max(frac, 1.0 / TOKENS)
    for _ in range(args.warmup):
        _oracle_fraction(h, frac, lib)
    nbytes = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        nbytes += _oracle_fraction(h, frac, lib)
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e9
    rows = max(1, int(round(TOKENS * frac)))
    sample = (f"each step: the first {rows} of {TOKENS} positions of every operator "
              f"(fp64 oracle, {cores} threads)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(STEP_CONFIG),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    del np
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ end to end

class SlabSet:
    """One step's tensors for the end-to-end leg, packed so that each direction is a single
    copy: the inputs (x, w, Q, K, sin, cos) are views of one device slab, the outputs (y,
    yQ, yK) of another; each view starts on a 256-byte boundary."""

    def __init__(self, src: InputSet):
        self.ins = self._pack(src.inputs_(), fill=True)
        self.outs = self._pack(src.outputs_(), fill=False)
        self.x, self.w, self.q, self.k, self.sq, self.cq = self.ins[1]
        self.y, self.yq, self.yk = self.outs[1]
        self.p = {n: getattr(self, n).data_ptr()
                  for n in ("x", "w", "q", "k", "sq", "cq", "y", "yq", "yk")}

    @staticmethod
    def _pack(tensors, fill: bool):
        offs, n = [], 0
        for t in tensors:
            offs.append(n)
            n += (t.numel() * t.element_size() + 255) // 256 * 256
        slab = torch.empty(n, dtype=torch.uint8, device="cuda")
        views = []
        for t, o in zip(tensors, offs):
            nb = t.numel() * t.element_size()
            v = slab[o:o + nb].view(t.dtype).view(t.shape)
            if fill:
                v.copy_(t)
            views.append(v)
        return slab, views


def _e2e_serial(sets, host_in, host_out, steps: int, stream) -> float:
    """Every step on one stream: copy in, the two kernels, copy out. Returns seconds."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record()
        for i in range(steps):
            s = sets[i % 2]
            s.ins[0].copy_(host_in, non_blocking=True)
            launch_step(s, stream.cuda_stream)
            host_out[i % 2].copy_(s.outs[0], non_blocking=True)
        e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e-3


def _e2e_pipelined(sets, host_in, host_out, steps: int) -> float:
    """Double-buffered over two device slab sets and three streams: the host-to-device copy
    of step i + 1, the kernels of step i and the device-to-host copy of step i - 1 run at
    the same time. Events keep each set's inputs from being overwritten before the kernels
    of its previous step have read them, and its outputs before they have been copied out.
    Returns seconds from the first copy in to the last copy out."""
    h2d, comp, d2h = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    in_ready = [ev(), ev()]
    comp_done = [ev(), ev()]
    out_done = [ev(), ev()]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(h2d)
    comp.wait_event(e0)
    d2h.wait_event(e0)
    for i in range(steps):
        k = i % 2
        s = sets[k]
        if i >= 2:
            h2d.wait_event(comp_done[k])     # step i - 2 has read this set's inputs
        with torch.cuda.stream(h2d):
            s.ins[0].copy_(host_in, non_blocking=True)
        in_ready[k].record(h2d)
        comp.wait_event(in_ready[k])
        if i >= 2:
            comp.wait_event(out_done[k])     # step i - 2's outputs have been copied out
        launch_step(s, comp.cuda_stream)
        comp_done[k].record(comp)
        d2h.wait_event(comp_done[k])
        with torch.cuda.stream(d2h):
            host_out[k].copy_(s.outs[0], non_blocking=True)
        out_done[k].record(d2h)
    e1.record(d2h)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e-3


def end_to_end(sets, steps: int, world: int, dist) -> dict:
    """The step metric through the C ABI with host buffers: each step copies its inputs
    from pinned host memory, runs both kernels and copies its outputs back to pinned host
    memory, all inside the timed region. Reported pipelined (the value) and serial."""
    slabs = [SlabSet(sets[0]), SlabSet(sets[1 % len(sets)])]
    host_in = slabs[0].ins[0].cpu().pin_memory()
    host_out = [torch.empty(slabs[0].outs[0].numel(), dtype=torch.uint8, pin_memory=True)
                for _ in range(2)]
    h2d = host_in.numel()
    d2h = host_out[0].numel()
    stream = torch.cuda.Stream()
    _e2e_serial(slabs, host_in, host_out, 3, stream)          # warm-up
    _e2e_pipelined(slabs, host_in, host_out, 3)
    if dist is not None:
        dist.barrier()
    t_pipe = _e2e_pipelined(slabs, host_in, host_out, steps)
    t_serial = _e2e_serial(slabs, host_in, host_out, steps, stream)
    t_pipe, t_serial = ranks_max([t_pipe, t_serial], dist)
    return {"value": job_value(STEP_BYTES, steps, world, t_pipe), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": t_pipe / steps * 1e3,
            "schedule": "double-buffered: copy in of step i+1, kernels of step i and copy out "
                        "of step i-1 on three streams, ordered by events; each direction one "
                        "copy of a packed slab (inputs, outputs 256-byte aligned in it)",
            "serial": {"value": job_value(STEP_BYTES, steps, world, t_serial),
                       "ms_per_step": t_serial / steps * 1e3,
                       "schedule": "one stream: copy in, kernels, copy out"},
            "copy_GB/s": (h2d + d2h) * steps / t_pipe / 1e9}


# ------------------------------------------------------------------ large configurations

def _kv_cat_tensors(B, P, S, Hk, D, n_rep, dt="bf16"):
    """Device inputs of one KV concat + repeat call: past, new, tables [P+S, D/2], output."""
    st = inputs.STORAGE[dt]
    past = torch.randn(B, P, Hk, D, device="cuda").to(st)
    new = torch.randn(B, S, Hk, D, device="cuda").to(st)
    _, sn, cs = inputs.rope_inputs(1, P + S, 1, D, dt, seed=0, device="cuda")
    out = torch.empty(B, P + S, Hk * n_rep, D, device="cuda", dtype=st)
    return past, new, sn, cs, out


LARGE_CASES = [
    ("rmsnorm fp32 [64,2048] (the small configuration; launch-bound)", "rms",
     (64, 2048, False, 1e-5, "f32")),
    ("rmsnorm bf16 [16384,8192] stress, eps 1e-6", "rms", (16384, 8192, True, 1e-6)),
    ("rmsnorm bf16 [65536,8192]", "rms", (65536, 8192, False, 1e-5)),
    ("rmsnorm bf16 [65536,3000]", "rms", (65536, 3000, False, 1e-5)),
    ("rmsnorm bf16 [65536,2048]", "rms", (65536, 2048, False, 1e-5)),
    ("add_rmsnorm bf16 [16384,8192]", "add", (16384, 8192)),
    ("add_rmsnorm bf16 [65536,2048]", "add", (65536, 2048)),
    ("rmsnorm bf16 [1024,65536] (staged in shared memory)", "rms", (1024, 65536, False, 1e-5)),
    ("rmsnorm bf16 [256,131072] (staged in shared memory)", "rms", (256, 131072, False, 1e-5)),
    ("add_rmsnorm bf16 [512,131072] (staged in shared memory)", "add", (512, 131072)),
    ("add_rmsnorm bf16 [2048,65536] (staged in shared memory)", "add", (2048, 65536)),
    ("layernorm bf16 [8192,4096]", "ln", (8192, 4096)),
    ("layernorm fp16 [8192,4096] (the TileLang tutorial's example 2)", "ln", (8192, 4096, "f16")),
    ("layernorm bf16 [65536,2048]", "ln", (65536, 2048)),
    ("layernorm bf16 [16384,8192]", "ln", (16384, 8192)),
    ("layernorm bf16 [1024,65536] (a cluster per row, chunks in shared memory)", "ln",
     (1024, 65536)),
    ("layernorm bf16 [256,131072] (a cluster per row, chunks in shared memory)", "ln",
     (256, 131072)),
    ("layernorm fp32 [1024,32768] (staged in shared memory, two rows a step)", "ln",
     (1024, 32768, "f32")),
    ("rmsnorm bf16 [1024,262152] (a cluster per row, chunks in shared memory)", "rms",
     (1024, 262152, False, 1e-5)),
    ("add_rmsnorm bf16 [256,300000] (a cluster per row, x and r in shared memory)", "add",
     (256, 300000)),
    ("layernorm bf16 [1024,262152] (a cluster per row, chunks in shared memory)", "ln",
     (1024, 262152)),
    ("layernorm bf16 [512,140000] (ragged staged chunks: a cluster per row)", "ln",
     (512, 140000)),
    ("rope bf16 [1,65536,32,128]", "rope", (65536, 32, 128)),
    ("rope fp16 [1,4096,32,128] (the TileLang tutorial's exercise E13)", "rope",
     (4096, 32, 128, "f16")),
    ("rope bf16 [1,65536,32,64]", "rope", (65536, 32, 64)),
    ("rope bf16 [1,65536,8,128]", "rope", (65536, 8, 128)),
    ("rope_qk bf16 Q[1,65536,32,128] + K[1,65536,8,128]", "rope_qk", (65536, 32, 8, 128)),
    ("kv rmsnorm+rope+cache bf16 kv[1,65536,512+64] -> 131072 slots", "kv", (65536, 512, 64)),
    ("rope interleaved bf16 x[65536,32,128], random positions < 131072", "ril", (65536, 32, 128)),
    ("kv cat + repeat bf16 K[8,8192,8,128] -> [8,8192,32,128], last 1024 rotated", "cat",
     (8, 7168, 1024, 8, 128, 4)),
    ("kv cat + repeat bf16 K[1,65536,8,64] -> [1,65536,32,64], last 4096 rotated", "cat",
     (1, 61440, 4096, 8, 64, 4)),
]


def _large_case(kind: str, shp: tuple, seed: int):
    """One input set of a large configuration: (launch(stream), bytes, kernel name, tensors).
    The launch closure keeps its own tensors alive; `tensors` is returned so that the
    caller can hold them across graph capture and replay as well."""
    if kind == "rms":
        rows, cols, stress, eps = shp[:4]
        dt = shp[4] if len(shp) > 4 else "bf16"
        x, w = inputs.rmsnorm_inputs(rows, cols, dt, seed=seed, stress=stress, device="cuda")
        y = torch.empty_like(x)
        pname = plan_name("rmsnorm", camp.camp_rmsnorm_plan(x, w, y, rows, cols, dt), dt)
        code = camp._dtype(dt)
        fn = lambda st: camp.camp_rmsnorm(x.data_ptr(), w.data_ptr(), y.data_ptr(), rows, cols,
                                          eps, code, st)
        return fn, ledger.rmsnorm_bytes(rows, cols, dt), pname, (x, w, y)
    if kind == "add":
        rows, cols = shp
        x, w = inputs.rmsnorm_inputs(rows, cols, "bf16", seed=seed, device="cuda")
        r, _ = inputs.rmsnorm_inputs(rows, cols, "bf16", seed=seed + 100, device="cuda")
        h, y = torch.empty_like(x), torch.empty_like(x)
        pname = "add_" + plan_name("rmsnorm", camp.camp_add_rmsnorm_plan(x, r, w, h, y, rows,
                                                                         cols, "bf16"))
        fn = lambda st: camp.camp_add_rmsnorm(x.data_ptr(), r.data_ptr(), w.data_ptr(),
                                              h.data_ptr(), y.data_ptr(), rows, cols, 1e-5,
                                              camp.BF16, st)
        return fn, ledger.add_rmsnorm_bytes(rows, cols), pname, (x, w, r, h, y)
    if kind == "ln":
        rows, cols = shp[:2]
        dt = shp[2] if len(shp) > 2 else "bf16"
        x, w, bt = inputs.layernorm_inputs(rows, cols, dt, seed=seed, device="cuda")
        y = torch.empty_like(x)
        pname = plan_name("layernorm", camp.camp_layernorm_plan(x, w, bt, y, rows, cols, dt), dt)
        code = camp._dtype(dt)
        fn = lambda st: camp.camp_layernorm(x.data_ptr(), w.data_ptr(), bt.data_ptr(),
                                            y.data_ptr(), rows, cols, 1e-5, code, st)
        return fn, ledger.layernorm_bytes(rows, cols, dt), pname, (x, w, bt, y)
    if kind == "ril":
        T, H, D = shp
        mp = 2 * T
        g = torch.Generator(device="cuda")
        g.manual_seed(seed)
        x = torch.randn(T, H, D, device="cuda", generator=g).to(torch.bfloat16)
        y = torch.empty_like(x)
        sn = torch.empty(mp, D // 2, device="cuda")
        cs = torch.empty(mp, D // 2, device="cuda")
        camp.camp_rope_tables(sn, cs, mp, D, THETA)
        pos = torch.randint(0, mp, (T,), device="cuda", dtype=torch.int32, generator=g)
        plan = camp.camp_rope_interleaved_plan(x, sn, cs, pos, y, T, H, D, mp, "bf16")
        pname = f"rope_interleaved<bf16,vec{plan.vec_bytes},hpt{plan.group}>"
        fn = lambda st: camp.camp_rope_interleaved(x.data_ptr(), sn.data_ptr(), cs.data_ptr(),
                                                   pos.data_ptr(), y.data_ptr(), T, H, D, mp,
                                                   camp.BF16, st)
        nbytes = 2 * T * H * D * 2 + 2 * T * (D // 2) * 4 + 4 * T
        return fn, nbytes, pname, (x, y, sn, cs, pos)
    if kind == "kv":
        S, Dn, Dr = shp
        ns = 2 * S
        g = torch.Generator(device="cuda")
        g.manual_seed(seed)
        x = torch.randn(1, S, Dn + Dr, device="cuda", generator=g).to(torch.bfloat16)
        gam = torch.ones(Dn, device="cuda", dtype=torch.bfloat16)
        _, sn, cs = inputs.rope_inputs(1, S, 1, Dr, "bf16", seed=seed, device="cuda")
        slots = torch.randperm(ns, device="cuda", generator=g)[:S].to(torch.int64)
        y = torch.empty(ns, Dn, device="cuda", dtype=torch.bfloat16)
        yr = torch.empty(ns, Dr, device="cuda", dtype=torch.bfloat16)
        plan = camp.camp_kv_rmsnorm_rope_cache_plan(x, gam, sn, cs, slots, y, yr, 1, S, Dn, Dr,
                                                    ns, "bf16")
        pname = f"kv_cache<bf16,vec{plan.vec_bytes},nv{plan.per_thread}>"
        fn = lambda st: camp.camp_kv_rmsnorm_rope_cache(
            x.data_ptr(), gam.data_ptr(), sn.data_ptr(), cs.data_ptr(), slots.data_ptr(),
            y.data_ptr(), yr.data_ptr(), 1, S, Dn, Dr, ns, 1e-5, camp.BF16, st)
        return fn, ledger.kv_cache_bytes(1, S, Dn, Dr), pname, (x, gam, sn, cs, slots, y, yr)
    if kind == "cat":
        B, P, S, Hk, D, nr = shp
        x, nw, sn, cs, y = _kv_cat_tensors(B, P, S, Hk, D, nr)
        plan = camp.camp_kv_cat_repeat_plan(x, nw, sn, cs, y, B, P, S, Hk, D, nr, "bf16")
        pname = f"kv_cat_repeat<bf16,vec{plan.vec_bytes},hpt{plan.group}>"
        fn = lambda st: camp.camp_kv_cat_repeat(x.data_ptr(), nw.data_ptr(), sn.data_ptr(),
                                                cs.data_ptr(), y.data_ptr(), B, P, S, Hk, D, nr,
                                                camp.BF16, st)
        return fn, ledger.kv_cat_repeat_bytes(B, P, S, Hk, D, nr), pname, (x, nw, sn, cs, y)
    if kind == "rope_qk":
        S, Hq, Hk, D = shp
        q, sn, cs = inputs.rope_inputs(1, S, Hq, D, "bf16", seed=seed, device="cuda")
        k, _, _ = inputs.rope_inputs(1, S, Hk, D, "bf16", seed=seed + 100, device="cuda")
        yq, yk = torch.empty_like(q), torch.empty_like(k)
        pname = plan_name("rope", camp.camp_rope_qk_plan(q, k, sn, cs, yq, yk, 1, S, Hq, Hk, D,
                                                         "bf16"))
        fn = lambda st: camp.camp_rope_qk(q.data_ptr(), k.data_ptr(), sn.data_ptr(),
                                          cs.data_ptr(), yq.data_ptr(), yk.data_ptr(), 1, S, Hq,
                                          Hk, D, camp.BF16, st)
        return fn, ledger.rope_qk_bytes(1, S, Hq, Hk, D), pname, (q, k, sn, cs, yq, yk)
    S, H, D = shp[:3]
    dt = shp[3] if len(shp) > 3 else "bf16"
    x, sn, cs = inputs.rope_inputs(1, S, H, D, dt, seed=seed, device="cuda")
    y = torch.empty_like(x)
    pname = plan_name("rope", camp.camp_rope_plan(x, sn, cs, y, 1, S, H, D, dt), dt)
    code = camp._dtype(dt)
    fn = lambda st: camp.camp_rope(x.data_ptr(), sn.data_ptr(), cs.data_ptr(), y.data_ptr(), 1,
                                   S, H, D, code, st)
    return fn, ledger.rope_bytes(1, S, H, D, dt), pname, (x, sn, cs, y)


SWEEP_TOKENS = (1, 8, 64, 512, 4096, 65536)


def sweep_cases() -> list:
    """The shape sweep: RMSNorm bf16 over tokens x hidden {2048, 3000, 8192} and RoPE bf16
    over tokens x heads {32, 8} x head_dim {64, 128} (B = 1, S = tokens, theta 500000)."""
    cases = []
    for t in SWEEP_TOKENS:
        for hidden in (2048, 3000, 8192):
            cases.append((f"rmsnorm bf16 [{t},{hidden}]", "rms", (t, hidden, False, 1e-5)))
        for heads in (32, 8):
            for d in (64, 128):
                cases.append((f"rope bf16 [1,{t},{heads},{d}]", "rope", (t, heads, d)))
    return cases


def case_rows(kind: str, shp: tuple) -> tuple[int, str]:
    """Rows a launch of this case processes, and what a row is: an RMSNorm / LayerNorm row,
    a (token, head) row of RoPE, a token of the KV kernels."""
    if kind in ("rms", "add", "ln"):
        return shp[0], "row"
    if kind in ("rope", "ril"):
        return shp[0] * shp[1], "head row"
    if kind == "rope_qk":
        return shp[0] * (shp[1] + shp[2]), "head row"
    if kind == "kv":
        return shp[0], "token"
    B, P, S = shp[:3]
    return B * (P + S), "token"


def oracle_case(kind: str, tensors: tuple, shp: tuple, budget_bytes: int = 64 << 20,
                runs: int = 5) -> dict | None:
    """CPU leg (the fp64 oracle, as it stands, on all host cores) of an RMSNorm or RoPE
    configuration: the median of `runs` calls on the first rows of its inputs (at most
    `budget_bytes` of input), as GB/s over the same algorithmic bytes and rows/s."""
    import numpy as np
    import oracle
    lib = oracle.load()
    cores = oracle.threads_available(lib)
    if kind == "rms":
        x, w = tensors[0], tensors[1]
        rows, cols, _, eps = shp[:4]
        dt = shp[4] if len(shp) > 4 else "bf16"
        n = max(1, min(rows, budget_bytes // (cols * x.element_size())))
        xs, ws = inputs.to_numpy(x[:n]), inputs.to_numpy(w)
        fn = lambda: oracle.rmsnorm(xs, ws, float(np.float32(eps)), dt, lib=lib)
        nbytes, what = ledger.rmsnorm_bytes(n, cols, dt), f"{n} of {rows} rows"
        nrows = n
    elif kind == "rope":
        x, sn, cs = tensors[0], tensors[1], tensors[2]
        S, H, D = shp[:3]
        dt = shp[3] if len(shp) > 3 else "bf16"
        n = max(1, min(S, budget_bytes // (H * D * x.element_size())))
        xs = inputs.to_numpy(x[:, :n])
        ss, cc = sn[:n].cpu().numpy(), cs[:n].cpu().numpy()
        fn = lambda: oracle.rope(xs, ss, cc, dt, lib=lib)
        nbytes, what = ledger.rope_bytes(1, n, H, D, dt), f"{n} of {S} positions"
        nrows = n * H
    else:
        return None
    fn()
    ts = []
    for _ in range(runs):
        t0 = time.perf_counter()
        fn()
        ts.append(time.perf_counter() - t0)
    t = statistics.median(ts)
    return {"GB/s": nbytes / t / 1e9, "rows_per_s": nrows / t, "cores": cores,
            "kind": "oracle", "sample": f"{what}, median of {runs}"}


# Most input sets one large-shape or sweep case rotates over: every case of at least
# 4 x L2 / MAX_SETS bytes (about 0.5 MB) is timed L2-cold.
MAX_SETS = 1024


def large_configs(peak: float, reps: int, cases=None, cpu: bool = False) -> list[dict]:
    """Single-operator timings, timed like the step: a CUDA graph of N back-to-back launches
    rotating over R input sets (R x bytes > 4 x L2 for every case of more than 4 x L2 /
    MAX_SETS bytes, so every launch reads from HBM), one event pair per graph replay; the
    median over `reps` replays of the replay time / N."""
    out = []
    l2 = getattr(torch.cuda.get_device_properties(torch.cuda.current_device()),
                 "L2_cache_size", 0) or 129 * 2**20
    for name, kind, shp in (LARGE_CASES if cases is None else cases):
        first = _large_case(kind, shp, 0)
        nbytes = first[1]
        R = max(1, min(MAX_SETS, math.ceil(4 * l2 / nbytes)))
        sets = [first] + [_large_case(kind, shp, i) for i in range(1, R)]
        N = R * max(1, round(16 / R))
        stream = torch.cuda.current_stream().cuda_stream
        for f in sets:
            f[0](stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        with torch.cuda.graph(g, stream=cap):
            h = torch.cuda.current_stream().cuda_stream
            for j in range(N):
                sets[j % R][0](h)
        g.replay()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]
        for a, b in evs:
            a.record()
            g.replay()
            b.record()
        torch.cuda.synchronize()
        t = statistics.median(a.elapsed_time(b) * 1e-3 for a, b in evs) / N
        gbs = nbytes / t / 1e9
        nrows, row_kind = case_rows(kind, shp)
        entry = {"config": name, "kernel": first[2], "bytes": nbytes, "us": t * 1e6,
                 "GB/s": gbs, "frac": gbs / peak, "rows_per_s": nrows / t, "row": row_kind,
                 "input_sets": R, "launches_per_graph": N, "l2_cold": R * nbytes > 4 * l2}
        if cpu and kind in ("rms", "rope"):
            entry["cpu_baseline"] = oracle_case(kind, first[3], shp)
        out.append(entry)
        del g, sets, first
        torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------ profiling cases

def parse_plan(text: str | None):
    """An explicit plan from `field=value,...` (the camp_plan_t fields), or None."""
    if not text:
        return None
    p = camp.Plan()
    for item in text.split(","):
        key, _, val = item.partition("=")
        if key not in dict(camp.Plan._fields_):
            raise SystemExit(f"unknown plan field {key!r}")
        setattr(p, key, int(val))
    return p


def run_case(case: str, launches: int, plan_text: str | None = None) -> None:
    """Launch one operator `launches` times at one shape (inputs drawn on the device),
    for profilers; prints the plan and the launch count. `case` is kind:AxBx..[:dtype]
    (dtype bf16 when left out); `plan_text` (rmsnorm and layernorm only) forces a plan."""
    forced = parse_plan(plan_text)
    kind, _, rest = case.partition(":")
    shape, _, dt = rest.partition(":")
    dt = dt or "bf16"
    code = camp._dtype(dt)
    st = inputs.STORAGE[dt]
    dims = [int(v) for v in shape.split("x")]
    torch.cuda.set_device(0)
    camp.load()
    stream = torch.cuda.current_stream().cuda_stream
    if kind == "rmsnorm":
        rows, cols = dims
        x, w = inputs.rmsnorm_inputs(rows, cols, dt, seed=0, device="cuda")
        y = torch.empty_like(x)
        plan = plan_name("rmsnorm", forced or camp.camp_rmsnorm_plan(x, w, y, rows, cols, dt), dt)
        for _ in range(launches):
            if forced is None:
                camp.camp_rmsnorm(x, w, y, rows, cols, EPS, code, stream)
            else:
                camp.camp_rmsnorm_with_plan(x, w, y, rows, cols, EPS, code, forced, stream)
    elif kind == "add":
        rows, cols = dims
        x, w = inputs.rmsnorm_inputs(rows, cols, dt, seed=0, device="cuda")
        r, _ = inputs.rmsnorm_inputs(rows, cols, dt, seed=1, device="cuda")
        h, y = torch.empty_like(x), torch.empty_like(x)
        plan = "add_" + plan_name("rmsnorm", camp.camp_add_rmsnorm_plan(x, r, w, h, y, rows, cols,
                                                                        dt), dt)
        for _ in range(launches):
            camp.camp_add_rmsnorm(x, r, w, h, y, rows, cols, EPS, code, stream)
    elif kind == "layernorm":
        rows, cols = dims
        x, w, bt = inputs.layernorm_inputs(rows, cols, dt, seed=0, device="cuda")
        y = torch.empty_like(x)
        plan = plan_name("layernorm", forced or camp.camp_layernorm_plan(x, w, bt, y, rows, cols, dt), dt)
        for _ in range(launches):
            if forced is None:
                camp.camp_layernorm(x, w, bt, y, rows, cols, EPS, code, stream)
            else:
                camp.camp_layernorm_with_plan(x, w, bt, y, rows, cols, EPS, code, forced, stream)
    elif kind == "rope_il":
        T, H, D = dims
        mp = 2 * T
        x = torch.randn(T, H, D, device="cuda").to(st)
        y = torch.empty_like(x)
        sn = torch.empty(mp, D // 2, device="cuda")
        cs = torch.empty(mp, D // 2, device="cuda")
        camp.camp_rope_tables(sn, cs, mp, D, THETA, stream)
        pos = torch.randint(0, mp, (T,), device="cuda", dtype=torch.int32)
        p = camp.camp_rope_interleaved_plan(x, sn, cs, pos, y, T, H, D, mp, dt)
        plan = f"rope_interleaved<{dt},vec{p.vec_bytes},hpt{p.group}>"
        for _ in range(launches):
            camp.camp_rope_interleaved(x, sn, cs, pos, y, T, H, D, mp, code, stream)
    elif kind == "kv":
        S, Dn, Dr = dims
        ns = 2 * S
        x = torch.randn(1, S, Dn + Dr, device="cuda").to(st)
        gam = torch.ones(Dn, device="cuda", dtype=st)
        _, sn, cs = inputs.rope_inputs(1, S, 1, Dr, dt, seed=0, device="cuda")
        slots = torch.randperm(ns, device="cuda")[:S].to(torch.int64)
        y = torch.empty(ns, Dn, device="cuda", dtype=st)
        yr = torch.empty(ns, Dr, device="cuda", dtype=st)
        p = camp.camp_kv_rmsnorm_rope_cache_plan(x, gam, sn, cs, slots, y, yr, 1, S, Dn, Dr, ns,
                                                 dt)
        plan = f"kv_cache<{dt},vec{p.vec_bytes},nv{p.per_thread}>"
        for _ in range(launches):
            camp.camp_kv_rmsnorm_rope_cache(x, gam, sn, cs, slots, y, yr, 1, S, Dn, Dr, ns, EPS,
                                            code, stream)
    elif kind == "kvcat":
        B, P, S, Hk, D, nr = dims
        x, nw, sn, cs, y = _kv_cat_tensors(B, P, S, Hk, D, nr, dt)
        p = camp.camp_kv_cat_repeat_plan(x, nw, sn, cs, y, B, P, S, Hk, D, nr, dt)
        plan = f"kv_cat_repeat<{dt},vec{p.vec_bytes},hpt{p.group}>"
        for _ in range(launches):
            camp.camp_kv_cat_repeat(x, nw, sn, cs, y, B, P, S, Hk, D, nr, code, stream)
    elif kind == "rope_qk":
        B, S, Hq, Hk, D = dims
        q, sn, cs = inputs.rope_inputs(B, S, Hq, D, dt, seed=0, device="cuda")
        k, _, _ = inputs.rope_inputs(B, S, Hk, D, dt, seed=1, device="cuda")
        yq, yk = torch.empty_like(q), torch.empty_like(k)
        plan = plan_name("rope", camp.camp_rope_qk_plan(q, k, sn, cs, yq, yk, B, S, Hq, Hk, D,
                                                        dt), dt)
        for _ in range(launches):
            camp.camp_rope_qk(q, k, sn, cs, yq, yk, B, S, Hq, Hk, D, code, stream)
    elif kind == "rope":
        B, S, H, D = dims
        x, sn, cs = inputs.rope_inputs(B, S, H, D, dt, seed=0, device="cuda")
        y = torch.empty_like(x)
        plan = plan_name("rope", camp.camp_rope_plan(x, sn, cs, y, B, S, H, D, dt), dt)
        for _ in range(launches):
            camp.camp_rope(x, sn, cs, y, B, S, H, D, code, stream)
    else:
        raise SystemExit(f"unknown case {case!r}")
    torch.cuda.synchronize()
    print(json.dumps({"case": case, "kernel": plan, "launches": launches}), flush=True)


# ------------------------------------------------------------------ the JSON line

def build_line(*, value: float, world: int, steps: int, warmup: int, ms_per_step: float,
               reps: int, M: int, kernels: list[dict], roofline: dict, cpu: dict | None,
               e2e: dict, clocks: dict, peak: float, detail_path: str | None) -> dict:
    """The one JSON line rank 0 prints last: the headline metric and the keys the
    benchmark contract names, and nothing bulky (the per-shape tables go to the detail
    file)."""
    r3 = lambda v: None if v is None else round(float(v), 3)
    short_k = [{"name": k["name"], "kernel": k["kernel"], "us": r3(k["us"]),
                "GB/s": r3(k["GB/s"]), "frac": r3(k["frac"])} for k in kernels]
    line = {
        "metric": METRIC, "value": r3(value), "unit": UNIT, "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": dict(STEP_CONFIG),
        "timing": {"repeats": reps, "stat": "median over repeats of the K-step region",
                   "graph_steps": M, "pct_of_peak": r3(100.0 * value / world / peak)},
        "roofline": {k: (r3(v) if isinstance(v, float) else v) for k, v in roofline.items()},
        "kernels": short_k,
        "cpu_baseline": None if cpu is None else {
            "value": r3(cpu["value"]), "unit": cpu["unit"], "cores": cpu["cores"],
            "kind": cpu["kind"], "sample": cpu["sample"]},
        "e2e": {"value": r3(e2e["value"]), "unit": e2e["unit"],
                "h2d_bytes_per_step": e2e["h2d_bytes_per_step"],
                "d2h_bytes_per_step": e2e["d2h_bytes_per_step"],
                "serial": r3(e2e["serial"]["value"])},
        "gpu_launches": len(kernels) * steps * reps,
        "clocks": {"sm_mhz": clocks.get("sm_mhz"), "sm_max_mhz": clocks.get("sm_max_mhz"),
                   "reasons": clocks.get("reasons", []), "samples": clocks.get("samples", 0)},
    }
    if detail_path:
        line["detail"] = detail_path
    return line


def line_text(line: dict) -> str:
    """The line as printed; raises if it is not under LINE_LIMIT bytes."""
    text = json.dumps(line, separators=(",", ":"))
    if len(text.encode()) > LINE_LIMIT:
        raise ValueError(f"the JSON line is {len(text)} bytes, over {LINE_LIMIT}")
    return text


def write_detail(path: str, detail: dict) -> str | None:
    try:
        os.makedirs(os.path.dirname(os.path.abspath(path)), exist_ok=True)
        with open(path, "w") as f:
            json.dump(detail, f, indent=1)
        return path
    except OSError as e:
        log(f"bench: could not write {path}: {e}")
        return None


# ------------------------------------------------------------------ the timed region

def make_flush(l2: int) -> torch.Tensor:
    """A buffer of twice the L2 size; reading it (flush_l2) evicts whatever a region left in
    L2. A read, not a write: a write would leave L2 full of dirty lines, whose write-back
    would then land inside the next timed region (about 126 MB of extra traffic, 8% of a
    20-step region)."""
    return torch.ones(2 * l2 // 4 + 1024, dtype=torch.float32, device="cuda")


def flush_l2(buf: torch.Tensor) -> None:
    torch.sum(buf)


def timing_event() -> torch.cuda.Event:
    """A timing event that, recorded during graph capture, becomes an event node of the
    graph (torch's `external` events); a plain timing event where torch lacks them."""
    try:
        return torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        return torch.cuda.Event(enable_timing=True)


def external_events_supported() -> bool:
    try:
        torch.cuda.Event(enable_timing=True, external=True)
        return True
    except TypeError:
        return False


class RegionBlock:
    """`count` consecutive steps (first, first + 1, ... on input sets mod R) as one CUDA
    graph: an event node, the steps' RMSNorm launches back to back, then their Q+K RoPE
    launches, and an event node at the end. The two operators of a step are independent,
    so a block runs all of its steps' work; consecutive launches overlap through
    programmatic dependent launch, the first RoPE launch after the last RMSNorm one
    included: the event that splits the two runs is recorded on a side branch of the graph
    (forked after the last RMSNorm launch, joined before the end), so it times that point
    without adding a dependency between the kernels. Without graph event nodes (older
    torch), the events are recorded between per-operator graphs instead."""

    def __init__(self, sets, first: int, count: int, in_graph: bool):
        self.in_graph = in_graph
        self.ev = [timing_event() for _ in range(len(KERNELS) + 1)]
        self.graphs = []
        cap = torch.cuda.Stream()
        # created before capture: the side stream and the fork/join events of each split
        sides = [(torch.cuda.Stream(), torch.cuda.Event(), torch.cuda.Event())
                 for _ in KERNELS[1:]]
        parts = [KERNELS] if in_graph else [(k,) for k in KERNELS]
        for part in parts:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                main = torch.cuda.current_stream()
                h = main.cuda_stream
                if in_graph:
                    self.ev[0].record()
                for ki, kind in enumerate(part):
                    for i in range(count):
                        launch(kind, sets[(first + i) % len(sets)], h)
                    if in_graph and ki + 1 < len(part):
                        side, fork, join = sides[ki]
                        fork.record(main)
                        side.wait_event(fork)
                        with torch.cuda.stream(side):
                            self.ev[ki + 1].record()
                        join.record(side)
                if in_graph:
                    for _, _, join in sides:
                        main.wait_event(join)
                if in_graph:
                    self.ev[len(part)].record()
            self.graphs.append(g)

    def replay(self) -> None:
        if self.in_graph:
            self.graphs[0].replay()
            return
        self.ev[0].record()
        for ki, g in enumerate(self.graphs):
            g.replay()
            self.ev[ki + 1].record()

    def times(self) -> list[float]:
        """Seconds of each operator's part in the last replay (after a synchronize)."""
        return [self.ev[i].elapsed_time(self.ev[i + 1]) * 1e-3 for i in range(len(KERNELS))]


def time_regions(blocks: list, reps: int, flush: torch.Tensor
                 ) -> tuple[list[float], dict[str, list[float]]]:
    """`reps` repeats of the K-step region (its blocks in order). Before each repeat L2 is
    flushed by a read, outside the events; after it the device is synchronized and the
    events read.
    Returns per repeat the region's seconds (first block's first event to the last block's
    last) and per operator the summed seconds of its parts."""
    region, per = [], {kind: [] for kind in KERNELS}
    for _ in range(reps):
        flush_l2(flush)
        for blk in blocks:
            blk.replay()
        torch.cuda.synchronize()
        region.append(blocks[0].ev[0].elapsed_time(blocks[-1].ev[-1]) * 1e-3)
        acc = [0.0] * len(KERNELS)
        for blk in blocks:
            for i, t in enumerate(blk.times()):
                acc[i] += t
        for kind, t in zip(KERNELS, acc):
            per[kind].append(t)
    return region, per


# ------------------------------------------------------------------ main

def main() -> None:
    ap = argparse.ArgumentParser(description="RMSNorm + RoPE hot-path benchmark")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=640)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--repeats", type=int, default=21,
                    help="least number of timed repeats of the K-step region (median reported)")
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="repeat the region until about this much GPU time (clock samples)")
    ap.add_argument("--impl", choices=("camp", "reference"), default="camp")
    ap.add_argument("--graph-steps", type=int, default=0,
                    help="steps per captured graph (0: up to 1024)")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=120.0)
    ap.add_argument("--large-reps", type=int, default=50)
    ap.add_argument("--detail", default=DETAIL_PATH,
                    help="file for the per-kernel, large-shape and sweep figures")
    ap.add_argument("--no-large", action="store_true", help="skip the large-shape timings")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--case", default=None,
                    help="profiling mode: launch one operator at one shape --launches times "
                         "and exit, e.g. rmsnorm:16384x8192, add:16384x8192, "
                         "layernorm:16384x2048, "
                         "rope:1x16384x32x128, rope_qk:1x16384x32x8x128 (B x S x Hq x Hk x D), "
                         "kv:65536x512x64 (S x Dn x Dr), rope_il:16384x32x128 (T x H x D, "
                         "random positions) or kvcat:1x3584x512x8x64x4 "
                         "(B x P x S x Hk x D x n_rep); a third field picks the storage "
                         "type, e.g. layernorm:8192x4096:f16 (bf16 when left out)")
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--plan", default=None,
                    help="with --case rmsnorm or layernorm: an explicit plan as camp_plan_t "
                         "fields, e.g. kernel=12,cluster=16,per_thread=2,rows_per_step=1")
    args = ap.parse_args()
    if args.case:
        run_case(args.case, args.launches, args.plan)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.steps < 1:
        ap.error("--steps must be at least 1")
    if args.repeats < 1:
        ap.error("--repeats must be at least 1")

    if args.impl == "reference":
        run_reference(args)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} needs {args.gpus} ranks (torchrun), found {world}")
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    camp.load()
    peak, peak_kind = load_peak()
    props = torch.cuda.get_device_properties(local)
    l2 = getattr(props, "L2_cache_size", 0) or 129 * 2**20
    R = max(2, math.ceil(4 * l2 / STEP_BYTES))
    sets = [InputSet(seed=rank * 1000 + i, device="cuda") for i in range(R)]
    flush = make_flush(l2)
    torch.cuda.synchronize()
    plans = {
        "rmsnorm": plan_name("rmsnorm", camp.camp_rmsnorm_plan(
            sets[0].x, sets[0].w, sets[0].y, TOKENS, HIDDEN, "bf16")),
        "rope_qk": plan_name("rope", camp.camp_rope_qk_plan(
            sets[0].q, sets[0].k, sets[0].sq, sets[0].cq, sets[0].yq, sets[0].yk, 1, TOKENS,
            HQ, HK, HEAD_DIM, "bf16")),
    }

    # Warm-up: W eager steps (also loads every kernel before capture).
    stream = torch.cuda.current_stream().cuda_stream
    for i in range(args.warmup):
        launch_step(sets[i % R], stream)
    torch.cuda.synchronize()

    M = min(args.graph_steps or 1024, args.steps)
    in_graph = external_events_supported()
    blocks = [RegionBlock(sets, s0, min(M, args.steps - s0), in_graph)
              for s0 in range(0, args.steps, M)]
    # Upload the graphs and size the repeats (untimed): at least --repeats, and enough for
    # about --min-seconds of GPU time so that the clock sampler sees the load.
    probe, _ = time_regions(blocks, 3, flush)
    t_rep = statistics.median(probe) + 2 * l2 / (peak * 1e9)
    reps = max(args.repeats, min(100000, math.ceil(args.min_seconds / max(t_rep, 1e-7))))
    reps = int(ranks_max([float(reps)], dist)[0])

    gpu_id = str(local)
    try:
        gpu_id = "GPU-" + str(props.uuid)
    except AttributeError:
        pass
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.5)

    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_host0 = time.time()
    region, per = time_regions(blocks, reps, flush)
    torch.cuda.synchronize()
    t_host1 = time.time()
    if dist is not None:
        dist.barrier()
    sampler.stop()
    clocks = sampler.summary(t_host0, t_host1)

    # The median repeat, then the slowest rank.
    elapsed = statistics.median(region)
    per_kernel = {kind: statistics.median(per[kind]) / args.steps for kind in KERNELS}
    maxed = ranks_max([elapsed] + [per_kernel[k] for k in KERNELS], dist)
    elapsed = maxed[0]
    per_kernel = dict(zip(KERNELS, maxed[1:]))

    value = job_value(STEP_BYTES, args.steps, world, elapsed)
    kernels = []
    for kind in KERNELS:
        t = per_kernel[kind]
        gbs = KERNEL_BYTES[kind] / t / 1e9
        rows = TOKENS if kind == "rmsnorm" else TOKENS * (HQ + HK)
        kernels.append({"name": kind, "kernel": plans[kind], "bytes": KERNEL_BYTES[kind],
                        "us": t * 1e6, "GB/s": gbs, "frac": gbs / peak, "rows_per_s": rows / t,
                        "row": "row" if kind == "rmsnorm" else "head row"})
    # Context only (another accelerator, not a target): the one throughput the pages print
    # for this operator and shape, RMSNorm bf16 4096 x 2048 counted as one read of x and one
    # write of y, 0.0707 ms = 474 GB/s (NineToothed backend on a MetaX C500).
    rms = next(k for k in kernels if k["name"] == "rmsnorm")
    xy_gbs = 2 * TOKENS * HIDDEN * 2 / (rms["us"] * 1e-6) / 1e9
    rms["published_context"] = {"GB/s": 474.0, "ms": 0.0707, "bytes": "x read + y write",
                                "hardware": "MetaX C500 (NineToothed backend)",
                                "this_kernel_same_bytes_GB/s": xy_gbs,
                                "ratio": xy_gbs / 474.0}
    dom = max(kernels, key=lambda k: k["us"])
    roofline = {"bound": "hbm", "achieved": dom["GB/s"], "peak": peak, "unit": "GB/s",
                "frac": dom["GB/s"] / peak, "traffic": recorded_traffic(dom["kernel"]),
                "kernel": dom["kernel"],
                "peak_source": "of measured (hbm_gbs)" if peak_kind == "measured"
                else "of fallback (6800 GB/s)"}

    # End to end through the C ABI with host buffers (pinned), copies inside the timing.
    e2e = end_to_end(sets, args.e2e_steps, world, dist)

    calibration = copy_calibration(sets, min(M, 64), 50, peak)
    del sets, blocks, flush
    torch.cuda.empty_cache()

    large = sweep = None
    if rank == 0 and not args.no_large:
        cpu_cases = world == 1 and not args.no_cpu
        large = large_configs(peak, args.large_reps, cpu=cpu_cases)
        sweep = large_configs(peak, args.large_reps, sweep_cases(), cpu=cpu_cases)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        s0 = InputSet(0, "cuda")
        cpu = cpu_baseline(_host_step_inputs(s0), args.cpu_seconds)
        del s0

    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return
    detail = {
        "metric": METRIC, "value": value, "unit": UNIT, "steps": args.steps,
        "repeats": reps, "region_seconds": region,
        "input_sets": R, "l2_bytes": l2,
        "timing": (f"{reps} repeats of the {args.steps}-step region, L2 flushed by a read "
                   f"before each; "
                   f"blocks of up to {M} steps, each "
                   + ("one CUDA graph with event nodes before and after the operators' "
                      "launch runs and one on a side branch between them" if in_graph else
                      "one CUDA graph per operator with events between them")
                   + "; per kernel: its summed time in the median repeat / K"),
        "kernels": kernels, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "clocks": clocks,
        "calibration": {"plain_copy_same_bytes": calibration,
                        "note": "device-to-device copies of each operator's bytes in the same "
                                "graph and rotation harness (outside the timed region): the "
                                "launch, ramp and drain cost any kernel of this size pays"},
        "large_configs": large, "sweep": sweep,
    }
    path = write_detail(args.detail, detail) if args.detail else None
    for group in (large or []) + (sweep or []):
        log(f"  {group['config']:<70s} {group['kernel']:<44s} {group['us']:9.2f} us "
            f"{group['GB/s']:8.1f} GB/s {group['frac']:.3f} cold={group['l2_cold']}")
    line = build_line(value=value, world=world, steps=args.steps, warmup=args.warmup,
                      ms_per_step=elapsed / args.steps * 1e3, reps=reps, M=M, kernels=kernels,
                      roofline=roofline, cpu=cpu, e2e=e2e, clocks=clocks, peak=peak,
                      detail_path=path)
    print(line_text(line), flush=True)


if __name__ == "__main__":
    main()
