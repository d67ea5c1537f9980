#!/usr/bin/env python3
"""Throughput of the sparse top-k MoE FFN layer's forward pass on GB300.

One step = one full forward pass of the layer (router + softmax + top-k, dispatch,
up-projection + GeLU, down-projection + gate, combine) over one batch of seeded
synthetic tokens, through the library's C ABI. Prints one JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

value      tokens/s of the whole job, device-timed with CUDA events over exactly K steps of
           moe_forward (inputs resident in HBM), max over ranks.
e2e        the same metric through the public layer object with the host->device copy of every
           step's tokens (pinned) and the device->host copy of its output inside the timed region,
           double-buffered: a step's copies overlap the neighbouring steps' compute.
roofline   the dominant kernel, timed live with CUDA events over back-to-back launches of its own
           C ABI call on the launching stream, against the measured peak in MEASURED_PEAKS.json.
cold_l2    context: one step at a time after a 512 MB scrub write (median of 20), the L2 cold.
cpu_baseline  the fp64 oracle on the host cores on a bounded prefix of the same batch.
--impl reference  the oracle alone, timed on the host cores, on the same workload and metric.

With N > 1 (torchrun) every rank runs its own replica of the layer on its own GPU with its own
batch (weak scaling, no collective on the data path).
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s; % of BF16 tensor peak (prefill) / % HBM BW (decode)"
DEFAULT_WORKLOAD = "skew_e128"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 126 * 2**20
TC_SOURCES = ["sparse_mixture_experts_moe_gb300/csrc/ffn_tc.cu", "sparse_mixture_experts_moe_gb300/csrc/common.cuh"]
TCT_SOURCES = ["sparse_mixture_experts_moe_gb300/csrc/ffn_tct.cu", "sparse_mixture_experts_moe_gb300/csrc/common.cuh"]
QUANT_SOURCES = ["sparse_mixture_experts_moe_gb300/csrc/quant.cu", "sparse_mixture_experts_moe_gb300/csrc/common.cuh"]
STREAM_SOURCES = ["sparse_mixture_experts_moe_gb300/csrc/ffn_stream.cu",
                  "sparse_mixture_experts_moe_gb300/csrc/common.cuh"]


def parse_args():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle sample")
    p.add_argument("--weight-bits", type=int, default=0, choices=[0, 4, 8],
                   help="0: the bf16 layer; 4 / 8: expert weights block-quantised to INT4 / INT8 (bf16 layers)")
    p.add_argument("--ffn-path", default="auto", choices=["auto", "tensor", "stream", "simt", "pair", "tensor_t"],
                   help="expert FFN kernel family (moe_path); auto = the library's own choice")
    p.add_argument("--also", default=None,
                   help="comma-separated extra workloads measured after the headline (graph replays, 20 steps) "
                        "and reported under 'other_workloads'; default: prefill_e128,decode_t64 when the "
                        "headline is the default workload, none otherwise; '' for none")
    p.add_argument("--launch", default="graph", choices=["graph", "direct"],
                   help="graph: replay a CUDA graph of the layer per step; direct: one C ABI call per kernel")
    return p.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def sources_sha(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def stored_traffic(kernel, workload, src_paths):
    """Per-launch DRAM bytes from the committed ncu summary, or None if absent or the kernel changed."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        entries = json.load(f)
    sha = sources_sha(src_paths)
    for e in entries:
        if e.get("kernel") == kernel and e.get("workload") == workload and e.get("source_sha256") == sha:
            return e.get("bytes_per_launch")
    return None


def workload_config(w, timing="CUDA events on the launching stream, max over ranks"):
    wbytes = w.E * 2 * w.d * w.F * (2 if w.dtype == 1 else 4)
    if wbytes > L2_BYTES:
        l2 = f"inputs larger than L2: {wbytes / 1e6:.0f} MB of expert weights vs {L2_BYTES / 2**20:.0f} MB L2"
    else:
        l2 = f"inputs fit in L2 ({wbytes / 1e6:.1f} MB of expert weights), no flush: a latency case"
    return {"workload": f"{w.name}: T={w.T} d={w.d} d_ff={w.F} E={w.E} top-{w.k}"
                        + (" skewed router bias" if w.skew else ""),
            "T": w.T, "d": w.d, "d_ff": w.F, "E": w.E, "k": w.k, "l2": l2, "timing": timing}


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest of every rank's value (the job's time is its slowest rank's); no-op for one rank."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank processes its own batch in the (max-over-ranks) step time."""
    return world * tokens_per_rank / (ms_per_step / 1e3)


# ----------------------------------------------------------------------------- inputs

def make_inputs(w, device, seed=0):
    import numpy as np
    import torch
    import inputgen as ig
    from inputgen import workloads
    tdt = torch.bfloat16 if w.dtype == ig.DTYPE_BF16 else torch.float32
    s = torch.cuda.current_stream().cuda_stream

    def fill(shape, stream_id, sigma):
        t = torch.empty(shape, dtype=tdt, device=device)
        ig.fill_device(t, 0, ig.stream_key(seed, stream_id), sigma, w.dtype, s)
        return t

    x = fill((w.T, w.d), ig.STREAM_X, 1.0)
    w_r = fill((w.d, w.E), ig.STREAM_WR, ig.sigma_for_fan_in(w.d))
    w1 = fill((w.E, w.d, w.F), ig.STREAM_W1, ig.sigma_for_fan_in(w.d))
    w2 = fill((w.E, w.F, w.d), ig.STREAM_W2, ig.sigma_for_fan_in(w.F))
    b_r = None
    c = workloads.bias_scale(w)
    if c is not None:
        b_r = torch.from_numpy(ig.skew_bias(w.E, c)).to(device)
    torch.cuda.synchronize()
    return x, w_r, b_r, w1, w2


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (host-stamped) of SM clock and throttle reasons while the GPU works."""
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap", "clocks.mem"]

    def __init__(self, gpu_index):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == len(self.FIELDS):
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        def pick(lo, hi):
            return [p for (t, p) in self.samples if lo <= t <= hi]
        win = pick(t0 - 0.15, t1 + 0.15)
        window = "timed region"
        if len(win) < 1:
            win = [p for (_, p) in self.samples]
            window = "whole GPU phase (timed region shorter than the 100 ms sampling period)"
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(p[0]) for p in win if num(p[0]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in win:
            for name, v in zip(names, p[4:8]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        mem = [num(p[8]) for p in win if num(p[8]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": num(win[0][1]),
                "mem_mhz": statistics.median(mem) if mem else None,
                "power_w_max": max((num(p[2]) or 0.0) for p in win), "reasons": sorted(reasons),
                "samples": len(win), "window": window}


# ----------------------------------------------------------------------------- CPU oracle

def host_copy(w, x, w_r, b_r, w1, w2, tokens):
    import numpy as np
    return dict(x=x[:tokens].double().cpu().numpy(), w_r=w_r.double().cpu().numpy(),
                b_r=None if b_r is None else b_r.double().cpu().numpy(),
                w1=HostExperts(w1), w2=HostExperts(w2))


class HostExperts:
    """Expert matrices as exact fp64 host arrays, copied once before any timing."""

    def __init__(self, t):
        self.t = t
        self.cache = {}

    def preload(self, experts):
        for e in experts:
            if e not in self.cache:
                self.cache[e] = self.t[e].double().cpu().numpy()

    def __getitem__(self, e):
        return self.cache[int(e)]


def oracle_sample(w, x, w_r, b_r, w1, w2, target_s, max_tokens=None, repeat=True):
    """Times oracle.forward on a prefix of the batch, or on the whole batch repeated when one pass is
    short of the target; returns (tokens/s, tokens per pass, seconds, cores, passes)."""
    import numpy as np
    import oracle
    cores = len(os.sched_getaffinity(0))
    max_tokens = w.T if max_tokens is None else min(max_tokens, w.T)
    # keep the fp64 copies of the touched experts within a sixth of the host's memory (at most 24 GB)
    per_expert = 2 * w.d * w.F * 8
    try:
        host_bytes = os.sysconf("SC_PAGE_SIZE") * os.sysconf("SC_PHYS_PAGES")
    except (ValueError, OSError, AttributeError):
        host_bytes = 36e9
    expert_budget = max(2, int(min(24e9, host_bytes / 6) // per_expert))
    n = min(max_tokens, 64 if w.E * per_expert > 6e9 else 256)
    h = host_copy(w, x, w_r, b_r, w1, w2, max_tokens)

    def run(ntok, passes=1):
        xs = h["x"][:ntok]
        idx = oracle.topk_select(oracle.router_logits(xs, h["w_r"], h["b_r"]), w.k)
        experts = sorted(set(int(e) for e in np.unique(idx)))
        if len(experts) > expert_budget:
            return None
        h["w1"].preload(experts)
        h["w2"].preload(experts)
        t0 = time.perf_counter()
        for _ in range(passes):
            oracle.forward(xs, h["w_r"], h["w1"], h["w2"], w.k, h["b_r"])
        return time.perf_counter() - t0

    dt = run(n)
    while dt is None and n > 1:
        n = max(1, n // 2)
        dt = run(n)
    if dt is None:
        raise RuntimeError("oracle sample: even one token touches more experts than the host budget")
    while dt < target_s / 4 and n < max_tokens:
        n2 = min(max_tokens, max(n + 1, int(n * min(8.0, target_s / max(dt, 1e-3)))))
        dt2 = run(n2)
        if dt2 is None:
            break
        n, dt = n2, dt2
    passes = 1
    if repeat and dt < target_s / 4:  # the sample is short (the whole batch, or all the experts the host
        passes = max(2, min(256, int(target_s / 2 / max(dt, 1e-3))))  # holds): repeat it
        dt = run(n, passes)
    return n * passes / dt, n, dt, cores, passes


# ----------------------------------------------------------------------------- our arm

def moved_routings(counts, reps):
    """Offsets [E+1] (int32) of routings 1, 2, ... that give the touched experts' rows, in expert order,
    to the experts i*s .. i*s + s - 1 (mod E), s = experts touched: the same rows and work per expert
    as the step's routing, on weights no neighbouring routing touches. Empty where E < 3 s."""
    import numpy as np
    counts = np.asarray(counts)
    E = counts.shape[0]
    held = counts[counts > 0]
    s = held.shape[0]
    out = []
    if s == 0 or E < 3 * s:
        return out
    for i in range(1, min(reps, E // s)):
        c = np.zeros(E, np.int64)
        c[(i * s + np.arange(s)) % E] = held
        out.append(np.concatenate([[0], np.cumsum(c)]).astype(np.int32))
    return out


def power_limited(clk):
    """Whether a clock record saw the power limit: sw_power_cap active, or the median SM clock under
    93% of its maximum."""
    if not clk or not clk.get("samples") or clk.get("window") != "timed region":
        return False  # no sample of the loop itself
    sm, top = clk.get("sm_mhz"), clk.get("sm_max_mhz")
    return "sw_power_cap" in clk.get("reasons", []) or (sm is not None and top and sm < 0.93 * top)


def dominant_roofline(w, kern_ms, touched, fpath, qbits, peaks, peak_src, kern_clk=None):
    """Roofline of the slower expert GEMM: algorithmic bytes (weight streaming) or FLOPs (tensor-core
    GEMMs) per launch over its measured launch time, against the measured peak. A tensor-core GEMM
    whose timing loop ran at the power limit is measured against the bf16 matmul rate sustained at
    that limit; one that kept its clocks, against the burst rate."""
    import sparse_mixture_experts_moe_gb300 as moe
    T, d, F, E, k, dt = w.T, w.d, w.F, w.E, w.k, w.dtype
    A = T * k
    eb = 2 if dt == 1 else 4
    dom = max(["expert_up", "expert_down"], key=lambda n: kern_ms[n])
    # the kernel family each GEMM ran (AUTO resolves per GEMM: moe_ffn_path)
    run_path = {n: (fpath if fpath != moe.PATH_AUTO else moe.ffn_path(T, k, E, F if n == "expert_up" else d, dt))
                for n in ("expert_up", "expert_down")}
    stream_path = run_path[dom] == moe.PATH_STREAM
    if qbits:
        # quantised weight streaming: codes + (scale, min) of the touched experts + rows in and out
        K_, N_ = (d, F) if dom == "expert_up" else (F, d)
        wbytes = K_ * N_ * qbits // 8 + (K_ // 64) * (N_ // 64) * 8
        alg_bytes = touched * wbytes + A * K_ * eb + A * N_ * (eb if dom == "expert_up" else 4)
        achieved = alg_bytes / (kern_ms[dom] / 1e3) / 1e9
        qname = f"ffn_stream_q{qbits}_kernel"
        qkey = f"{qname}<{1 if dom == 'expert_up' else 2}>"
        roof = {"kernel": f"{qname} ({dom})", "bound": "hbm", "achieved": achieved,
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                "traffic": stored_traffic(qkey, w.name, QUANT_SOURCES),
                "alg_bytes_per_launch": alg_bytes, "ms_per_launch": kern_ms[dom],
                "peak_source": f"{peak_src} hbm_gbs"}
    elif stream_path:
        # weight streaming: bytes = touched experts' matrix + the routed rows in and out
        if dom == "expert_up":
            alg_bytes = touched * d * F * eb + A * d * eb + A * F * eb
        else:
            alg_bytes = touched * F * d * eb + A * F * eb + A * d * eb
        achieved = alg_bytes / (kern_ms[dom] / 1e3) / 1e9
        roof = {"kernel": f"ffn_stream_tma_kernel ({dom})", "bound": "hbm", "achieved": achieved,
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                "traffic": stored_traffic(f"ffn_stream_tma_kernel<{1 if dom == 'expert_up' else 2}>", w.name,
                                          STREAM_SOURCES),
                "alg_bytes_per_launch": alg_bytes, "ms_per_launch": kern_ms[dom],
                "peak_source": f"{peak_src} hbm_gbs"}
    else:
        alg_flops = 2.0 * A * d * F
        achieved = alg_flops / (kern_ms[dom] / 1e3) / 1e12
        clk = (kern_clk or {}).get(dom)
        sustained = power_limited(clk)
        peak = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
        if sustained:
            why = (f"bf16_tflops_sustained (the launch's timing loop ran at the power limit: "
                   f"SM median {clk.get('sm_mhz')} MHz, {', '.join(clk.get('reasons', [])) or 'no reason'})")
        else:
            why = "bf16_tflops (burst: the launch's timing loop kept its clocks)"
        kname = {moe.PATH_TENSOR_PAIR: "ffn_tc2_kernel", moe.PATH_TENSOR_T: "ffn_tct_kernel"}.get(run_path[dom],
                                                                                               "ffn_tc_kernel")
        # attainable: min(peak, arithmetic intensity x HBM bandwidth), the intensity over the bytes the
        # GEMM must move (touched experts' weights, rows in, rows out)
        K_, N_ = (d, F) if dom == "expert_up" else (F, d)
        must_bytes = touched * K_ * N_ * eb + A * K_ * eb + A * N_ * (eb if dom == "expert_up" else 4)
        attainable = min(peak, alg_flops / must_bytes * peaks["hbm_gbs"] / 1e3)
        roof = {"kernel": f"{kname} ({dom})", "bound": "tensor", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "attainable": attainable,
                "frac_of_attainable": achieved / attainable,
                "traffic": stored_traffic(f"{kname}<{1 if dom == 'expert_up' else 2}>", w.name,
                                          TCT_SOURCES if kname == "ffn_tct_kernel" else TC_SOURCES),
                "alg_flops_per_launch": alg_flops, "ms_per_launch": kern_ms[dom],
                "peak_source": f"{peak_src} {why}",
                "frac_of_burst": achieved / peaks["bf16_tflops"],
                "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                "timing_loop_clocks": clk}
    return roof



def run_ours(args, w, rank, world, device):
    import numpy as np
    import torch
    import torch.distributed as dist
    import sparse_mixture_experts_moe_gb300 as moe

    x, w_r, b_r, w1, w2 = make_inputs(w, device, seed=rank)
    T, d, F, E, k, dt = w.T, w.d, w.F, w.E, w.k, w.dtype
    A = T * k
    out = torch.empty_like(x)
    ws = torch.empty(moe.workspace_bytes(T, d, F, E, k, dt), dtype=torch.uint8, device=device)
    moe.workspace_init(ws)
    stream = torch.cuda.current_stream()

    qbits = args.weight_bits
    fpath = {"auto": moe.PATH_AUTO, "tensor": moe.PATH_TENSOR, "stream": moe.PATH_STREAM, "simt": moe.PATH_SIMT,
             "pair": moe.PATH_TENSOR_PAIR, "tensor_t": moe.PATH_TENSOR_T}[args.ffn_path]
    q1 = q2 = None
    if qbits:
        if dt != 1:
            raise SystemExit("--weight-bits needs a bf16 workload")
        q1, q2 = moe.quantize(w1, qbits), moe.quantize(w2, qbits)  # once, before timing
        torch.cuda.synchronize()

    def direct_step(s=None):
        if qbits:
            moe.forward_q(x, w_r, b_r, q1, q2, T, d, F, E, k, qbits, out, ws, stream=s)
        else:
            moe.forward(x, w_r, b_r, w1, w2, T, d, F, E, k, dt, out, ws, path=fpath, stream=s)

    graph = None
    if args.launch == "graph":
        # the layer's kernels captured once (moe_graph_capture_begin / _end); each step replays all of them
        with moe.GraphCapture(keep=(x, w_r, b_r, w1, w2, out, ws, q1, q2)) as cap:
            direct_step(cap.stream)
        graph = cap.graph

        def step():
            graph.launch(stream)
    else:
        step = direct_step

    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                          else os.environ["CUDA_VISIBLE_DEVICES"].split(",")[torch.cuda.current_device()])
    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()
    st, detail = moe.get_device_status(ws)
    if st != moe.MOE_OK:
        raise RuntimeError(f"device status after warm-up: {moe.status_string(st)} ({detail})")

    # --- timed region: exactly K steps of moe_forward
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        dist.barrier()
    ms_total = max_over_ranks(ev0.elapsed_time(ev1), world, device)
    ms_per_step = ms_total / args.steps
    value = job_tokens_per_s(T, world, ms_per_step)

    # --- context: the same K steps as one host call per kernel (no graph)
    ms_direct = None
    if graph is not None:
        for _ in range(3):
            direct_step()
        torch.cuda.synchronize()
        ed0, ed1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ed0.record(stream)
        for _ in range(args.steps):
            direct_step()
        ed1.record(stream)
        torch.cuda.synchronize()
        ms_direct = max_over_ranks(ed0.elapsed_time(ed1), world, device) / args.steps

    # --- context: steps on a cold L2. Before each, a 512 MB buffer (four times the L2) is written on
    # the same stream; only the step lies between the two events. The median of 20 is reported.
    scrub = torch.empty(512 * 2**20 // 4, dtype=torch.float32, device=device)
    cold = []
    ec0, ec1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(20):
        scrub.fill_(float(i))
        ec0.record(stream)
        step()
        ec1.record(stream)
        torch.cuda.synchronize()
        cold.append(ec0.elapsed_time(ec1))
    ms_cold = float(np.median(cold))
    del scrub

    # --- per-kernel timing: the step as its separate C ABI calls (dispatch: the two-kernel public entry)
    idx = torch.empty((T, k), dtype=torch.int32, device=device)
    gate = torch.empty((T, k), dtype=torch.float32, device=device)
    counts = torch.empty(E, dtype=torch.int32, device=device)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=device)
    perm = torch.empty(A, dtype=torch.int32, device=device)
    row_of = torch.empty((T, k), dtype=torch.int32, device=device)
    row_gate = torch.empty(A, dtype=torch.float32, device=device)
    x_perm = torch.empty((A, d), dtype=x.dtype, device=device)
    h = torch.empty((A, F), dtype=x.dtype, device=device)
    y_perm = torch.empty((A, d), dtype=torch.float32, device=device)
    # Each kernel is launched R times back to back between two events on the launching stream, so
    # the host's per-call work (argument marshalling, tensor maps) overlaps the previous launch and
    # only device time is measured; repeated calls on the same inputs give the same outputs.
    reps = max(args.steps, 10)
    moe.router_topk(x, w_r, b_r, T, d, E, k, dt, idx, gate)
    moe.dispatch(x, idx, gate, T, d, E, k, dt, counts, offsets, perm, row_of, row_gate, x_perm, ws)
    counts_h = counts.cpu().numpy()
    touched = int((counts_h > 0).sum())
    # An expert GEMM whose touched weights fit in twice the L2 would find part of them there when
    # repeated on the same experts. Launch i then gives the touched experts' rows, in order, to the
    # experts i*s .. i*s + s - 1 (mod E; s = experts touched), so that neighbouring launches read
    # weights that none near them has read. The shape of the work is unchanged.
    w_bytes = touched * d * F * (qbits / 8 if qbits else (2 if dt == 1 else 4))
    routings = [offsets]
    if w_bytes < 2 * L2_BYTES:
        routings += [torch.from_numpy(o).to(device) for o in moved_routings(counts_h, reps)]
    kernel_timing = ("back-to-back launches; the expert GEMMs' rows moved to other experts at every launch "
                     f"({len(routings)} routings) because the touched weights fit in twice the L2"
                     if len(routings) > 1 else "back-to-back launches on the step's routing")

    def up_call(i=0):
        offs = routings[i % len(routings)]
        if qbits:
            moe.expert_up_q(x_perm, q1[0], q1[1], offs, T, d, F, E, k, qbits, h)
        else:
            moe.expert_up(x_perm, w1, offs, T, d, F, E, k, dt, h, ws, path=fpath)

    def down_call(i=0):
        offs = routings[i % len(routings)]
        if qbits:
            moe.expert_down_q(h, q2[0], q2[1], offs, row_gate, T, d, F, E, k, qbits, y_perm)
        else:
            moe.expert_down(h, w2, offs, row_gate, T, d, F, E, k, dt, y_perm, ws, path=fpath)

    calls = [("router_topk", lambda i=0: moe.router_topk(x, w_r, b_r, T, d, E, k, dt, idx, gate)),
             ("dispatch", lambda i=0: moe.dispatch(x, idx, gate, T, d, E, k, dt, counts, offsets, perm, row_of,
                                                   row_gate, x_perm, ws)),
             ("expert_up", up_call), ("expert_down", down_call),
             ("combine", lambda i=0: moe.combine(y_perm, row_of, T, d, k, dt, out))]
    kern_ms, kern_wall = {}, {}
    for name, fn in calls:
        fn()  # warm-up, and the inputs of the next kernel (on the step's own routing)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        tw0 = time.time()
        ev0.record(stream)
        for i in range(reps):
            fn(i)
        ev1.record(stream)
        torch.cuda.synchronize()
        kern_wall[name] = (tw0, time.time())
        kern_ms[name] = ev0.elapsed_time(ev1) / reps

    # --- e2e: public layer object, pinned host tokens in, output back to the host, every step.
    # Double-buffered as a serving loop runs it: step i's input copy (its own stream) overlaps step
    # i-1's compute, and step i's output copy (a third stream) overlaps step i+1's compute; events
    # keep a buffer from being refilled before the step that used it has finished with it.
    layer = moe.MoELayer(w_r, w1, w2, k=k, b_r=b_r, path=fpath, weight_bits=qbits or None)
    x_host = x.cpu().pin_memory()
    out_host = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(x) for _ in range(2)]
    out_dev = [torch.empty_like(out) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)
    if graph is not None:
        layer_graphs = [layer.graph(x_dev[b], out_dev[b]) for b in range(2)]

        def layer_step(b):
            layer_graphs[b].launch(stream)
    else:
        def layer_step(b):
            with torch.cuda.stream(stream):
                layer(x_dev[b], out=out_dev[b])
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_steps(n):
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_comp[b])        # step i-2 has read x_dev[b]
                x_dev[b].copy_(x_host, non_blocking=True)
                ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])           # step i-2's output has left out_dev[b]
            layer_step(b)
            ev_comp[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[b])
                out_host[b].copy_(out_dev[b], non_blocking=True)
                ev_out[b].record(s_out)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)

    e2e_steps(4)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    e2e_steps(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_value = job_tokens_per_s(T, world, max_over_ranks(e0.elapsed_time(e1) / args.steps, world, device))
    st, detail = moe.get_device_status(ws)
    if st != moe.MOE_OK:
        raise RuntimeError(f"device status after timing: {moe.status_string(st)} ({detail})")
    clocks.stop()
    clk = clocks.summary(t_wall0, t_wall1)
    # the clocks of each GEMM's own timing loop: they choose between the burst and sustained peaks
    kern_clk = {n: clocks.summary(*kern_wall[n]) for n in ("expert_up", "expert_down")}

    # --- roofline of the dominant kernel
    peaks, peak_src = load_peaks()
    roof = dominant_roofline(w, kern_ms, touched, fpath, qbits, peaks, peak_src, kern_clk)

    result = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if dt == 1 else "f32", "data": "synthetic (seeded inputgen draws)",
        "config": dict(workload_config(w), parallelism=f"replicas x{world}" if world > 1 else "single GPU",
                       weights=(f"INT{qbits} codes, 64x64 blocks with fp32 (scale, min), quantised once before "
                                "timing" if qbits else "bf16" if dt == 1 else "fp32"),
                       ffn_path=args.ffn_path,
                       launch=("CUDA graph of the layer's kernels (moe_forward_graph_create), one graph launch "
                               "per step" if graph is not None else "one C ABI call per kernel")),
        "ms_per_step_direct_calls": ms_direct,
        "cold_l2": {"ms_per_step": ms_cold, "value": job_tokens_per_s(T, world, ms_cold),
                    "how": "each step alone after writing a 512 MB buffer on its stream, median of 20"},
        "roofline": roof,
        "kernel_ms": kern_ms,
        "kernel_timing": kernel_timing,
        "experts_touched": touched,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": x.numel() * x.element_size(),
                "d2h_bytes_per_step": out.numel() * out.element_size(),
                "copies": "every step, double-buffered on their own streams (overlapping neighbouring steps)"},
        "gpu_launches": moe.forward_launches(T, d, F, E, k, dt, moe.PATH_STREAM if qbits else fpath) * args.steps,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not qbits:
        v, n, secs, cores, passes = oracle_sample(w, x, w_r, b_r, w1, w2, args.cpu_seconds)
        result["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                  "sample": (f"first {n} of the batch's {T} tokens (as many as the host holds "
                                             "the touched experts of, in fp64)" if n < T else
                                             f"the batch's {T} tokens") + ", fp64 oracle forward" +
                                            (f", {passes} passes" if passes > 1 else "") + f", {secs:.2f} s"}
    return result


def measure_extra(name, device, steps=20, warmup=3, reps=10):
    """One more workload beside the headline: device-timed graph replays of the layer (inputs resident,
    weights larger than L2), tokens/s, and the roofline of its slower expert GEMM."""
    import torch
    import sparse_mixture_experts_moe_gb300 as moe
    from inputgen import workloads
    w = workloads.get(name)
    x, w_r, b_r, w1, w2 = make_inputs(w, device)
    T, d, F, E, k, dt = w.T, w.d, w.F, w.E, w.k, w.dtype
    A = T * k
    out = torch.empty_like(x)
    ws = torch.empty(moe.workspace_bytes(T, d, F, E, k, dt), dtype=torch.uint8, device=device)
    moe.workspace_init(ws)
    stream = torch.cuda.current_stream()
    with moe.GraphCapture(keep=(x, w_r, b_r, w1, w2, out, ws)) as cap:
        moe.forward(x, w_r, b_r, w1, w2, T, d, F, E, k, dt, out, ws, stream=cap.stream)
    for _ in range(warmup):
        cap.graph.launch(stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        cap.graph.launch(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    idx = torch.empty((T, k), dtype=torch.int32, device=device)
    gate = torch.empty((T, k), dtype=torch.float32, device=device)
    counts = torch.empty(E, dtype=torch.int32, device=device)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=device)
    perm = torch.empty(A, dtype=torch.int32, device=device)
    row_of = torch.empty((T, k), dtype=torch.int32, device=device)
    row_gate = torch.empty(A, dtype=torch.float32, device=device)
    x_perm = torch.empty((A, d), dtype=x.dtype, device=device)
    h = torch.empty((A, F), dtype=x.dtype, device=device)
    y_perm = torch.empty((A, d), dtype=torch.float32, device=device)
    moe.router_topk(x, w_r, b_r, T, d, E, k, dt, idx, gate)
    moe.dispatch(x, idx, gate, T, d, E, k, dt, counts, offsets, perm, row_of, row_gate, x_perm, ws)
    kern_ms = {}
    for name_, fn in [("expert_up", lambda: moe.expert_up(x_perm, w1, offsets, T, d, F, E, k, dt, h, ws)),
                      ("expert_down", lambda: moe.expert_down(h, w2, offsets, row_gate, T, d, F, E, k, dt, y_perm,
                                                              ws))]:
        fn()
        torch.cuda.synchronize()
        k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        k0.record(stream)
        for _ in range(reps):
            fn()
        k1.record(stream)
        torch.cuda.synchronize()
        kern_ms[name_] = k0.elapsed_time(k1) / reps
    st, detail = moe.get_device_status(ws)
    if st != moe.MOE_OK:
        raise RuntimeError(f"device status ({name}): {moe.status_string(st)} ({detail})")
    touched = int((counts > 0).sum().item())
    peaks, peak_src = load_peaks()
    roof = dominant_roofline(w, kern_ms, touched, moe.PATH_AUTO, 0, peaks, peak_src)
    res = {"workload": workload_config(w)["workload"], "value": T / (ms / 1e3), "unit": "tokens/s",
           "ms_per_step": ms, "steps": steps, "warmup": warmup, "kernel_ms": kern_ms, "experts_touched": touched,
           "roofline": roof}
    del x, w_r, w1, w2, ws, out, x_perm, h, y_perm
    torch.cuda.empty_cache()
    return res


# ----------------------------------------------------------------------------- reference arm

def run_reference(args, w):
    """The fp64 oracle on the host cores: K timed steps (after W untimed), each a bounded prefix of the batch."""
    import torch
    import oracle
    device = "cuda" if torch.cuda.is_available() else "cpu"
    if device == "cuda":
        x, w_r, b_r, w1, w2 = make_inputs(w, device)
    else:
        x, w_r, b_r, w1, w2 = _cpu_inputs(w)
    budget_per_step = 150.0 / max(1, args.steps + args.warmup)
    v, n, secs, cores, passes = oracle_sample(w, x, w_r, b_r, w1, w2, min(args.cpu_seconds, budget_per_step),
                                              repeat=False)
    h = host_copy(w, x, w_r, b_r, w1, w2, n)
    import numpy as np
    idx = oracle.topk_select(oracle.router_logits(h["x"], h["w_r"], h["b_r"]), w.k)
    experts = sorted(set(int(e) for e in np.unique(idx)))
    h["w1"].preload(experts)
    h["w2"].preload(experts)
    for _ in range(args.warmup):
        oracle.forward(h["x"], h["w_r"], h["w1"], h["w2"], w.k, h["b_r"])
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.forward(h["x"], h["w_r"], h["w1"], h["w2"], w.k, h["b_r"])
    secs = (time.perf_counter() - t0) / max(1, args.steps)
    value = n / secs
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded inputgen draws)",
        "config": workload_config(w, timing="host wall clock (time.perf_counter) around K oracle steps"),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"first {n} of the batch's {w.T} tokens per step, fp64 oracle forward"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def _cpu_inputs(w):
    import torch
    import inputgen as ig
    from inputgen import workloads
    if w.E * w.d * w.F > (1 << 27):
        raise RuntimeError("reference arm without a GPU supports only small workloads")
    tdt = torch.bfloat16 if w.dtype == ig.DTYPE_BF16 else torch.float32

    def draw(shape, sid, sigma):
        import numpy as np
        n = int(np.prod(shape))
        a = ig.draw(0, n, ig.stream_key(0, sid), sigma, w.dtype)
        t = torch.from_numpy(a.view(np.int16) if w.dtype == ig.DTYPE_BF16 else a)
        return (t.view(torch.bfloat16) if w.dtype == ig.DTYPE_BF16 else t).reshape(shape)
    x = draw((w.T, w.d), ig.STREAM_X, 1.0)
    w_r = draw((w.d, w.E), ig.STREAM_WR, ig.sigma_for_fan_in(w.d))
    w1 = draw((w.E, w.d, w.F), ig.STREAM_W1, ig.sigma_for_fan_in(w.d))
    w2 = draw((w.E, w.F, w.d), ig.STREAM_W2, ig.sigma_for_fan_in(w.F))
    c = workloads.bias_scale(w)
    b_r = None if c is None else torch.from_numpy(ig.skew_bias(w.E, c))
    return x, w_r, b_r, w1, w2


def main():
    args = parse_args()
    from inputgen import workloads
    w = workloads.get(args.workload)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, w)), flush=True)
        return 0
    import torch
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    res = run_ours(args, w, rank, world, device)
    also = args.also if args.also is not None else (
        "prefill_e128,decode_t64" if args.workload == DEFAULT_WORKLOAD and world == 1 else "")
    extra = [n for n in also.split(",") if n]
    if extra:
        import gc
        gc.collect()
        torch.cuda.empty_cache()
        res["other_workloads"] = {n: measure_extra(n, device) for n in extra}
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
