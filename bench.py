#!/usr/bin/env python
"""Throughput of the Mamba-2 SSD chunked forward at the Mamba-2 2.7B layer shape.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one pass of the whole hot path -- chunk cumsum, chunk states, state
pass, fused output -- over one batch of the workload (b=8, T=4096, H=80, P=64,
N=128, G=1, L=256, bf16; x is 335 MB, larger than L2, so nothing is flushed
between steps).  Inputs are seeded synthetic tensors, resident in HBM before
the timed region.  Each step is one whole-path call through the C ABI
(mamba2_ssd_fwd, the call a user makes); every EVENT_EVERY-th step goes through
mamba2_ssd_fwd_timed (the same kernels, launched strictly one after another)
and records CUDA events between its stages on the launching stream, so the
per-kernel times and the whole-step time come from the same timed region.
(Events between kernels cost device time and rule out the overlapped launches
of stages 2-4; on every step they would add ~3 % to it.)

Printed (one JSON line, rank 0): tokens/s (value), TFLOP/s, per-kernel times,
the roofline of the dominant kernel, the whole-path roofline under the fixed
four-stage byte model, an end-to-end figure through ssd_fwd with host buffers
(H2D and D2H inside the timed region), SM clocks sampled during the timed
region, and the fp64 oracle timed on the host cores on a bounded sample.

--impl reference times the oracle (the reference arm of this method: a plain
CPU fp64 recurrence) on the same workload, metric and unit.

Other modes (one JSON line each, not the step above): --decode times the
single-token decode step on the workload's state (a CUDA graph of 8 steps);
--backward times mamba2_ssd_bwd on the workload; --all-configs prints the
whole-path forward on every measured workload (median per-call device time,
L2 flushed between calls where the inputs fit in it; on tensor-core shapes the
same call forced onto the CUDA-core kernels is timed beside it).

Multi-GPU (torchrun, N > 1): each rank runs its own batch of the workload
(independent (b, h) problems, no collective on the data path): weak scaling.
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SSD fwd tokens/s & TFLOP/s at Mamba-2 2.7B shape; % of roofline on 1 GB300"
EVENT_EVERY = 8                    # stage events on every 8th timed step
KERNELS_FUSED = ("chunk_cumsum", "chunk_state_pass", "chunk_out")
KERNELS_SPLIT = ("chunk_cumsum", "chunk_state", "state_pass", "chunk_out")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="mamba2-2.7b",
                    help="mamba2-2.7b (default), long-prefill, grouped-init")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--decode", action="store_true",
                    help="time the single-token decode step on the workload's state instead")
    ap.add_argument("--all-configs", action="store_true",
                    help="print one JSON line per measured workload (forward whole path): "
                         "median per-call device time, L2 flushed between calls when the "
                         "inputs fit in it")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward pass (mamba2_ssd_bwd) on the workload instead")
    ap.add_argument("--fused-state", action="store_true",
                    help="time stages 2+3 as the one fused kernel (mamba2_ssd_chunk_state_pass)")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch (smaller cases for profiler captures)")
    ap.add_argument("--seqlen", type=int, default=0,
                    help="override the workload's sequence length (profiler captures)")
    ap.add_argument("--nheads", type=int, default=0,
                    help="override the workload's head count, a multiple of its groups "
                         "(profiler captures)")
    return ap.parse_args()


def workload(name):
    from mamba_ssd_chunked_02_gb300 import workloads as W
    return {"mamba2-2.7b": W.MAMBA2_2P7B, "long-prefill": W.LONG_PREFILL,
            "grouped-init": W.GROUPED_INIT}[name]


# ----------------------------------------------------------- algorithmic model ---
def model(w, dsz=4):
    """Algorithmic bytes and tensor FLOPs per launch of each stage (dS moved
    between stages 2 and 3 with dsz bytes per element), and the whole-path
    figures (fixed four-stage byte model with fp32 states)."""
    b, T, H, P, N, G, L = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups, w.chunk_size
    E = 2 if w.dtype == "bf16" else 4
    nc = -(-T // L)
    th = b * T * H                        # token-heads
    st = b * nc * H * P * N               # per-chunk state elements
    init = 1 if w.init_std > 0 else 0
    k = {
        "chunk_cumsum": dict(bytes=12 * th + 4 * H, flops=0),
        "chunk_state": dict(bytes=th * (P * E + 8) + b * T * G * N * E + dsz * st,
                            flops=2 * th * P * N),
        "state_pass": dict(bytes=dsz * st + E * st + 4 * b * H * P * N * (1 + init) + 4 * b * H * nc,
                           flops=0),
        # stages 2+3 in one kernel: no dS round trip (the carried state moves
        # between CTAs through L2 and is not counted)
        "chunk_state_pass": dict(bytes=th * (P * E + 8) + b * T * G * N * E + E * st +
                                 4 * b * H * P * N * (1 + init),
                                 flops=2 * th * P * N),
        "chunk_out": dict(bytes=th * (2 * P * E + 8) + 2 * b * T * G * N * E + E * st + 4 * H,
                          flops=b * T * (H * (2 * P * N + P * (L + 1)) + G * N * (L + 1))),
    }
    graded = b * T * (H * (3 * P * E + 28 + 16 * P * N / L) + 3 * G * N * E) + \
        4 * b * H * P * N * (1 + init)
    flops = b * T * (H * (4 * P * N + P * (L + 1)) + G * N * (L + 1))
    return k, graded, flops


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def traffic_from_profile(kernel, w):
    """DRAM bytes per launch recorded with the committed ncu summary of this kernel
    and workload (profiles/<kernel>_<workload>.json), or None when absent or taken
    on a different kernel source."""
    tag = w.name.split()[0]
    path = os.path.join(ROOT, "profiles", f"{kernel}_{tag}.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as fh:
            fields = json.load(fh)
        src = fields["source"]
        want = fields["source_sha256_16"]
        traffic = float(fields["traffic_bytes_per_launch"])
    except (OSError, ValueError, KeyError, TypeError):
        return None
    spath = os.path.join(ROOT, src)
    if not os.path.exists(spath) or hashlib.sha256(open(spath, "rb").read()).hexdigest()[:16] != want:
        return None
    return traffic


def io_floor(w):
    """Bytes a single fused kernel would have to move at least: read x, dt, B, C
    once, write y once, plus the state I/O (final_state, and the initial state
    when given); no intermediate in HBM."""
    b, T, H, P, N, G = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    E = 2 if w.dtype == "bf16" else 4
    init = 1 if w.init_std > 0 else 0
    return b * T * (H * (2 * P * E + 4) + 2 * G * N * E) + 4 * b * H * P * N * (1 + init)


# --------------------------------------------------------------------- clocks ---
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            self.t0 = time.time()
        except Exception:
            self.proc = None

    def mark(self):
        return time.time()

    def stop(self, t_begin, t_end):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as fh:
            for i, line in enumerate(fh):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        # -lms 100: row i was taken about 0.1*i s after start; keep the rows of the
        # timed region (with one sample of slack either side).
        span = [r for i, r in enumerate(rows)
                if t_begin - 0.15 <= self.t0 + 0.1 * i <= t_end + 0.15] or rows
        def num(v):
            try:
                return float(v)
            except ValueError:
                return float("nan")
        sm = [num(r[1]) for r in span]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in span:
            for name, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": num(span[0][2]),
                "reasons": sorted(reasons), "samples": len(span),
                "power_w_max": max(num(r[3]) for r in span)}


# ------------------------------------------------------------------ CPU legs ---
def oracle_sample(inp, w, npairs, nthreads=0):
    """Time the fp64 recurrent oracle, as it stands, on `npairs` (b=0, h) pairs."""
    import oracle
    sl = {k: (v[:1] if v is not None and k in ("x", "dt", "B", "C", "initial_state") else v)
          for k, v in inp.items()}
    pairs = [(0, h % w.nheads) for h in range(npairs)]
    t0 = time.perf_counter()
    oracle.ssd_recurrent(**sl, ngroups=w.ngroups, pairs=pairs, nthreads=nthreads)
    return time.perf_counter() - t0


def cpu_baseline(inp, w, budget_s=15.0):
    import oracle
    cores = oracle.max_threads()
    t1 = oracle_sample(inp, w, cores)                  # one pair per thread: calibration
    rounds = max(1, int(budget_s / max(t1, 1e-3)))
    npairs = min(cores * rounds, 16 * w.nheads * w.batch)
    t = oracle_sample(inp, w, npairs)
    tokens = npairs * w.seqlen / w.nheads               # (b, h) pairs -> layer tokens
    return {"value": tokens / t, "unit": "tokens/s", "cores": min(cores, npairs),
            "kind": "oracle",
            "sample": f"fp64 recurrent oracle on {npairs} (batch, head) pairs x {w.seqlen} tokens "
                      f"of {w.name} ({npairs / w.nheads:.2f} layer-sequences), {t:.1f} s"}


def run_reference(args, w):
    import oracle
    from mamba_ssd_chunked_02_gb300 import workloads as W
    inp = W.make_inputs(w.scaled(batch=1))
    cores = oracle.max_threads()
    for _ in range(args.warmup):
        oracle_sample(inp, w, cores)
    times = [oracle_sample(inp, w, cores) for _ in range(args.steps)]
    t = sum(times)
    tokens = args.steps * cores * w.seqlen / w.nheads
    val = tokens / t
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * t / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, args.gpus),
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: fp64 recurrent oracle on {cores} (batch, head) "
                                   f"pairs x {w.seqlen} tokens of {w.name}"},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------- multi-rank host ---
def rank_workload(w, rank):
    """The problem rank `rank` runs: the same shape, its own batch of sequences
    (inputs drawn from seed + rank), so ranks share no data and need no collective."""
    return w.scaled(seed=w.seed + rank)


def max_over_ranks(value, dist, device):
    """A time measured on every rank -> the slowest rank's (the job's) time."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens(w, world):
    """Tokens the whole job processes per step (weak scaling: one batch per rank)."""
    return w.tokens * world


def config_of(w, n):
    return {"workload": w.name, "batch": w.batch, "seq_len": w.seqlen, "nheads": w.nheads,
            "headdim": w.headdim, "dstate": w.dstate, "ngroups": w.ngroups,
            "chunk_size": w.chunk_size, "io_dtype": w.dtype,
            "l2": "inputs larger than L2 (x alone is larger), no flush",
            "parallelism": "replicas" if n == 1 else f"dp{n}: one batch per rank, no collective"}


# ------------------------------------------------------------------- GPU leg ---
def run_decode(args, w):
    """Decode step (mamba2_ssd_decode) on the workload's (b, H, P, N) state: one
    token per sequence per step; an HBM stream of the state (read + write).
    Steps are replayed from a CUDA graph of eight launches, one per rotating state,
    as a decoding loop runs them; the Python binding's per-call argument checks
    (several microseconds) would otherwise be timed instead of the kernel."""
    import torch
    import mamba_ssd_chunked_02_gb300 as m2
    from mamba_ssd_chunked_02_gb300 import workloads as W
    wd = w.scaled(seqlen=1, init_std=0.1)
    inp = W.make_inputs(wd)
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    b, H, P, N, G = wd.batch, wd.nheads, wd.headdim, wd.dstate, wd.ngroups
    states = [dev["initial_state"].clone() for _ in range(8)]   # 8 x 21 MB > L2: no flush needed
    x, dt, B, C = dev["x"][:, 0], dev["dt"][:, 0], dev["B"][:, 0], dev["C"][:, 0]
    y = torch.empty((b, H, P), dtype=x.dtype, device="cuda")
    cs = torch.cuda.Stream()
    with torch.cuda.stream(cs):
        for i in range(8):
            m2.ssd_decode(states[i], x, dt, dev["A"], B, C, dev["D"], y=y, stream=cs)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cs):
        for i in range(8):
            m2.ssd_decode(states[i], x, dt, dev["A"], B, C, dev["D"], y=y, stream=cs)
    stream = torch.cuda.current_stream()
    for _ in range(max(3, args.warmup)):
        graph.replay()
    torch.cuda.synchronize()
    reps = max(1, (args.steps + 7) // 8)
    K = 8 * reps
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    clocks.start()
    time.sleep(0.3)
    wall0 = time.time()
    a.record(stream)
    for _ in range(reps):
        graph.replay()
    z.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop(wall0, time.time())
    if m2.device_error() != 0:
        raise RuntimeError("device-side error in the decode loop")
    ms = a.elapsed_time(z) / K
    E = 2 if wd.dtype == "bf16" else 4
    nbytes = 8 * b * H * P * N + b * H * (2 * P * E + 4) + 2 * b * G * N * E
    pk, src = peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    print(json.dumps({
        "metric": "SSD decode step: tokens/s (one token per sequence) at the workload's state",
        "value": b / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16" if wd.dtype == "bf16" else "f32",
        "data": "synthetic", "config": {"workload": wd.name, "batch": b, "nheads": H, "headdim": P,
                                         "dstate": N, "ngroups": G,
                                         "l2": "8 rotating states of 21 MB (> L2 together)",
                                         "launch": "CUDA graph of 8 decode steps, replayed"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / pk["hbm_gbs"], "traffic": None, "kernel": "decode",
                     "algorithmic_bytes": nbytes},
        "gpu_launches": K, "clocks": clk}), flush=True)


def run_all_configs(args):
    """Every measured workload through mamba2_ssd_fwd: each call timed alone with
    CUDA events on the launching stream; when the workload's inputs and outputs
    fit in L2 twice over, a 512 MB buffer is written between calls (outside the
    timed region), so every call starts with cold inputs."""
    import torch
    import mamba_ssd_chunked_02_gb300 as m2
    from mamba_ssd_chunked_02_gb300 import workloads as W
    pk, src = peaks()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    for w in W.ALL:
        inp = W.make_inputs(w)
        dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
        sh = m2.shape_of(dev["x"], dev["B"], w.chunk_size, w.ngroups)
        sh_cc = m2.shape_of(dev["x"], dev["B"], w.chunk_size, w.ngroups, m2.FLAG_FORCE_SIMT)
        ws = torch.empty(max(1, m2.workspace_size(sh), m2.workspace_size(sh_cc)),
                         dtype=torch.uint8, device="cuda")
        y = torch.empty_like(dev["x"])
        fin = torch.empty((w.batch, w.nheads, w.headdim, w.dstate), device="cuda")
        E = 2 if w.dtype == "bf16" else 4
        io = (2 * w.batch * w.seqlen * w.nheads * w.headdim + 2 * w.batch * w.seqlen * w.ngroups *
              w.dstate) * E
        cold = io < 2 * (129 << 20)

        def timed(flags):
            def call():
                m2.ssd_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                           dev["initial_state"], chunk_size=w.chunk_size, ngroups=w.ngroups,
                           y=y, final_state=fin, workspace=ws, flags=flags)

            for _ in range(max(3, args.warmup)):
                call()
            torch.cuda.synchronize()
            ts = []
            for _ in range(max(5, min(args.steps, 50))):
                if cold:
                    flush.fill_(1)
                a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                call()
                z.record(stream)
                z.synchronize()
                ts.append(a.elapsed_time(z))
            if m2.device_error() != 0:
                raise RuntimeError(f"device-side error on {w.name}")
            return sorted(ts)[len(ts) // 2], len(ts)

        tc = m2.path(sh) == m2.PATH_TCGEN05
        ms, calls = timed(0)
        # A bf16 whole-path call with 64-token chunks on a tensor-core shape runs
        # as 128-token chunks (same y and final state, half the chunk states):
        # grade it against the byte model of the chunk length it runs.
        wm = w.scaled(chunk_size=128) if tc and w.chunk_size == 64 else w
        _, graded, flops = model(wm)
        t_path = max(graded / (pk["hbm_gbs"] * 1e9), flops / (pk["bf16_tflops"] * 1e12))
        line = {"workload": w.name, "ms": ms, "tokens_per_s": w.tokens / (ms * 1e-3),
                "tflops": flops / (ms * 1e-3) / 1e12, "path_roofline_ms": t_path * 1e3,
                "path_frac": t_path / (ms * 1e-3), "peaks": src,
                "path": "tcgen05" if tc else "simt", "model_chunk_size": wm.chunk_size,
                "l2": "flushed between calls" if cold else "inputs larger than L2",
                "calls": calls}
        if tc:
            # the same call on the CUDA-core kernels, for comparison
            line["cuda_core_ms"] = timed(m2.FLAG_FORCE_SIMT)[0]
        print(json.dumps(line), flush=True)
        del dev, ws, y, fin
        torch.cuda.empty_cache()


def bwd_bytes(w):
    """Fixed HBM byte model of one backward call: read x and dy, write dx (fp32);
    read dt, write ddt; read B and C, write dB and dC (fp32); the chunk states
    handed between kernels counted at fp32 twice (the recomputed forward's dS /
    Sprev and the adjoint pass's dSout / Gn: 16 P N / L bytes per token-head
    each); read dfinal, write dinit (and read the initial state) when present."""
    b, T, H, P, N, G, L = (w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups,
                           w.chunk_size)
    E = 2 if w.dtype == "bf16" else 4
    init = 1 if w.init_std > 0 else 0
    per_th = 2 * P * E + 4 * P + 8 + 2 * 16 * P * N / L
    per_tg = 2 * N * E + 8 * N
    return b * T * (H * per_th + G * per_tg) + 4 * b * H * P * N * (1 + 2 * init)


def bwd_flops(w):
    """Contraction work of the backward: the forward's (chunk states, C.B^T,
    the intra-chunk and carried-state products) three more times over -- the
    reversed output run for dx, and the two transposed-state runs for dC and
    dB -- plus the chunk adjoints (2 P N per token-head); causal halves."""
    b, T, H, P, N, G, L = (w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups,
                           w.chunk_size)
    fwd = T * (H * (4 * P * N + P * (L + 1)) + G * N * (L + 1))
    return b * (4 * fwd + T * H * 2 * P * N)


def run_backward(args, w):
    """Backward pass (mamba2_ssd_bwd) on the workload, inputs and incoming gradients
    resident in HBM; reported against a fixed HBM byte model of the backward."""
    import torch
    import mamba_ssd_chunked_02_gb300 as m2
    from mamba_ssd_chunked_02_gb300 import workloads as W
    inp = W.make_inputs(w)
    gr = W.make_grads(w)
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    dy, dfin = gr["dy"].cuda(), gr["dfinal"].cuda()
    sh = m2.shape_of(dev["x"], dev["B"], w.chunk_size, w.ngroups)
    ws = torch.empty(m2.bwd_workspace_size(sh), dtype=torch.uint8, device="cuda")
    grads = None

    def step():
        nonlocal grads
        grads = m2.ssd_bwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                           dev["initial_state"], dy, dfin, chunk_size=w.chunk_size,
                           ngroups=w.ngroups, grads=grads, workspace=ws)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    K = args.steps
    stream = torch.cuda.current_stream()
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    clocks.start()
    time.sleep(0.3)
    wall0 = time.time()
    a.record(stream)
    for _ in range(K):
        step()
    z.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop(wall0, time.time())
    if m2.device_error() != 0:
        raise RuntimeError("device-side error in the backward loop")
    ms = a.elapsed_time(z) / K
    F = bwd_flops(w)
    nbytes = bwd_bytes(w)
    pk, src = peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    print(json.dumps({
        "metric": "SSD backward: tokens/s", "value": w.tokens / (ms * 1e-3), "unit": "tokens/s",
        "n_gpus": 1, "steps": K, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic", "config": dict(config_of(w, 1), what="backward, forward recompute included",
                                            grads="fp32"),
        "tflops": F / (ms * 1e-3) / 1e12,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / pk["hbm_gbs"], "traffic": None, "kernel": "whole backward",
                     "model": "backward I/O + chunk states at fp32 twice (bench.bwd_bytes)",
                     "algorithmic_bytes": nbytes, "peak_source": src},
        # 10 of the library's kernels per call on the tensor-core path: stages 1-3
        # (recompute), the y run, the chunk adjoints, bwd_state_pass_rev, the y' run,
        # dC, dB, bwd_token (plus two memsets)
        "gpu_launches": 10 * K, "clocks": clk}), flush=True)


def main():
    args = parse_args()
    w = workload(args.workload)
    if args.batch > 0:
        w = w.scaled(batch=args.batch, name=w.name.replace(f" b{w.batch} ", f" b{args.batch} "))
    if args.seqlen > 0:
        w = w.scaled(seqlen=args.seqlen, name=w.name.replace(f" T{w.seqlen} ", f" T{args.seqlen} "))
    if args.nheads > 0:
        if args.nheads % w.ngroups:
            raise SystemExit("--nheads must be a multiple of the workload's groups")
        w = w.scaled(nheads=args.nheads, name=w.name.replace(f" H{w.nheads} ", f" H{args.nheads} "))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            run_reference(args, w)
        return

    import torch
    import mamba_ssd_chunked_02_gb300 as m2
    from mamba_ssd_chunked_02_gb300 import workloads as W

    torch.cuda.set_device(local)
    if args.decode:
        if rank == 0:
            run_decode(args, w)
        return
    if args.backward:
        if rank == 0:
            run_backward(args, w)
        return
    if args.all_configs:
        if rank == 0:
            run_all_configs(args)
        return
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    inp_cpu = W.make_inputs(rank_workload(w, rank))
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp_cpu.items()}
    b, T, H, P, N = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate
    sh = m2.shape_of(dev["x"], dev["B"], w.chunk_size, w.ngroups)
    f32 = dict(dtype=torch.float32, device="cuda")
    fused = args.fused_state and m2.chunk_state_pass_workspace_size(sh) > 0
    KERNELS = KERNELS_FUSED if fused else KERNELS_SPLIT
    flags = m2.FLAG_FUSED_STATE if fused else 0
    y = torch.empty((b, T, H, P), dtype=w.torch_dtype, device="cuda")
    fin = torch.empty((b, H, P, N), **f32)
    ws = torch.empty(m2.workspace_size(sh), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    # event k of a step: before stage 1 (k = 0) and after stages 1..4 (k = 1..4)
    bounds = (0, 1, 3, 4) if fused else (0, 1, 2, 3, 4)

    def step(ev=None):
        """One step = one whole-path call (mamba2_ssd_fwd, or _fwd_timed with events)."""
        m2.ssd_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                   dev["initial_state"], chunk_size=w.chunk_size, ngroups=w.ngroups, y=y,
                   final_state=fin, workspace=ws, stream=stream, flags=flags, events=ev)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if m2.device_error() != 0:
        raise RuntimeError("device-side error during warm-up")

    K = args.steps
    timed = list(range(0, K, EVENT_EVERY))     # steps that record stage events
    evs = {i: [torch.cuda.Event(enable_timing=True) for _ in range(5)] for i in timed}
    for e in evs.values():         # create the CUDA events before the timed region
        for x_ in e:
            x_.record(stream)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.time()
    t_start.record(stream)
    for i in range(K):
        step(evs.get(i))
    t_end.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    if dist:
        dist.barrier()
    clk = clocks.stop(wall0, wall1)
    if m2.device_error() != 0:
        raise RuntimeError("device-side error in the timed region")

    total_ms = max_over_ranks(t_start.elapsed_time(t_end), dist, "cuda")
    ms_step = total_ms / K
    per = {k: 0.0 for k in KERNELS}
    for e in evs.values():
        for j, kname in enumerate(KERNELS):
            per[kname] += e[bounds[j]].elapsed_time(e[bounds[j + 1]])
    per = {k: v / len(evs) for k, v in per.items()}

    # the whole-path call hands dS from stage 2 to 3 in bf16 on the tensor-core path
    kmodel, graded_bytes, flops = model(w, 2 if m2.path(sh) == m2.PATH_TCGEN05 else 4)
    pk, pk_src = peaks()
    tokens = job_tokens(w, world)
    value = tokens / (ms_step * 1e-3)

    dom = max(per, key=per.get)
    dm = kmodel[dom]
    t_dom = per[dom] * 1e-3
    hbm_time = dm["bytes"] / (pk["hbm_gbs"] * 1e9)
    tc_time = dm["flops"] / (pk["bf16_tflops"] * 1e12) if dm["flops"] else 0.0
    if hbm_time >= tc_time:
        roof = {"bound": "hbm", "achieved": dm["bytes"] / t_dom / 1e9, "peak": pk["hbm_gbs"],
                "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": dm["flops"] / t_dom / 1e12,
                "peak": pk["bf16_tflops"], "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    tr = traffic_from_profile(dom, w)
    roof.update({"traffic": tr, "kernel": dom, "algorithmic_bytes": dm["bytes"],
                 "algorithmic_flops": dm["flops"], "ms": per[dom],
                 "timed_launches": len(evs),     # launches inside the timed region with events around them
                 "peak_source": f"{pk_src} (MEASURED_PEAKS.json)" if pk_src == "measured"
                 else "fallback"})

    t_path = max(graded_bytes / (pk["hbm_gbs"] * 1e9), flops / (pk["bf16_tflops"] * 1e12))
    # Three byte counts for the same measured step: the graded four-stage model
    # (dS and Sprev at fp32), the bytes the path's kernels are specified to move
    # (the sum of the per-kernel models, with its actual hand-off types), and the
    # I/O floor of a single fused kernel.
    moved = sum(kmodel[k]["bytes"] for k in KERNELS)
    floor = io_floor(w)
    hbm = pk["hbm_gbs"] * 1e9
    path_roof = {"model": "four-stage HBM hand-off, dS and Sprev counted at fp32",
                 "graded_bytes": graded_bytes, "flops": flops, "roofline_ms": t_path * 1e3,
                 "frac": t_path / (ms_step * 1e-3),
                 "bytes_moved": moved, "bytes_moved_frac": moved / hbm / (ms_step * 1e-3),
                 "io_floor_bytes": floor, "io_floor_frac": floor / hbm / (ms_step * 1e-3)}
    kernels = {}
    for kname in KERNELS:
        km = kmodel[kname]
        tk = per[kname] * 1e-3
        kernels[kname] = {"ms": per[kname], "GB/s": km["bytes"] / tk / 1e9,
                          "TFLOP/s": km["flops"] / tk / 1e12,
                          "hbm_frac": km["bytes"] / tk / 1e9 / pk["hbm_gbs"]}

    # End to end through ssd_fwd with pinned host buffers: every step copies its
    # inputs in (H2D) and its outputs y and final_state out (D2H).  Steps are
    # pipelined as a serving loop would run them: step i+1's inputs go in and step
    # i-1's outputs come out on two copy streams while step i computes, with two
    # device copies of every input and output.
    e2e = None
    if not args.no_e2e:
        host_in = {k: (v.pin_memory() if v is not None else None) for k, v in inp_cpu.items()}
        y_host = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for _ in range(2)]
        f_host = [torch.empty(fin.shape, dtype=fin.dtype).pin_memory() for _ in range(2)]
        din = [dev, {k: (torch.empty_like(v) if v is not None else None) for k, v in dev.items()}]
        ydev = [y, torch.empty_like(y)]
        fdev = [fin, torch.empty_like(fin)]
        h2d = sum(v.numel() * v.element_size() for v in host_in.values() if v is not None)
        d2h = y_host[0].numel() * y_host[0].element_size() + f_host[0].numel() * f_host[0].element_size()
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

        def run_e2e(n):
            ev_in = [torch.cuda.Event() for _ in range(n)]
            ev_comp = [torch.cuda.Event() for _ in range(n)]
            ev_out = [torch.cuda.Event() for _ in range(n)]
            a = torch.cuda.Event(enable_timing=True)
            z = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            s_in.wait_event(a)
            s_out.wait_event(a)
            for i in range(n):
                j = i & 1
                with torch.cuda.stream(s_in):          # inputs of step i
                    if i >= 2:
                        s_in.wait_event(ev_comp[i - 2])   # step i-2 is done reading them
                    for k, v in host_in.items():
                        if v is not None:
                            din[j][k].copy_(v, non_blocking=True)
                    ev_in[i].record(s_in)
                stream.wait_event(ev_in[i])            # compute of step i
                if i >= 2:
                    stream.wait_event(ev_out[i - 2])   # step i-2's outputs are out
                d = din[j]
                m2.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["initial_state"],
                           chunk_size=w.chunk_size, ngroups=w.ngroups, y=ydev[j],
                           final_state=fdev[j], workspace=ws, stream=stream, flags=flags)
                ev_comp[i].record(stream)
                with torch.cuda.stream(s_out):         # outputs of step i
                    s_out.wait_event(ev_comp[i])
                    y_host[j].copy_(ydev[j], non_blocking=True)
                    f_host[j].copy_(fdev[j], non_blocking=True)
                    ev_out[i].record(s_out)
            stream.wait_event(ev_out[n - 1])
            z.record(stream)
            torch.cuda.synchronize()
            return a.elapsed_time(z)

        run_e2e(3)
        ke = max(2, args.e2e_steps)
        if dist:
            dist.barrier()
        ems = max_over_ranks(run_e2e(ke), dist, "cuda")
        if m2.device_error() != 0:
            raise RuntimeError("device-side error in the end-to-end loop")
        e2e = {"value": tokens / (ems / ke * 1e-3), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": ke,
               "ms_per_step": ems / ke,
               "pipelined": "H2D of step i+1 and D2H of step i-1 overlap step i"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(inp_cpu, w)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
            "config": config_of(w, world),
            "tflops": flops * world / (ms_step * 1e-3) / 1e12,
            "roofline": roof, "path_roofline": path_roof, "kernels": kernels,
            "path": "tcgen05" if m2.path(sh) == m2.PATH_TCGEN05 else "simt",
            "gpu_launches": len(KERNELS) * K, "e2e": e2e, "cpu_baseline": cpu, "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
