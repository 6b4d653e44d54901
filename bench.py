"""Benchmark of the FLASH mixed-chunk attention forward core on GB300.

One step = one forward pass of the whole core (chunk states, chunk-axis scan,
chunk attention with the U gate) over one batch of synthetic input, through
the C ABI.  Default workload: the long causal shape (B=2, n=8192, C=256,
s=128, e=1536, bf16 I/O, fp32 accumulation).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

Prints one JSON line (rank 0).  Our arm: `value` is tokens/s over K steps with
inputs resident in HBM, timed with CUDA events on the launching stream between
a barrier + synchronize on both sides (max over ranks); per-kernel durations
come from events the library records between its kernels.  Inputs and outputs
rotate over three buffer sets, each larger than L2 (129 MB) for the default
workload, so no step reads what the previous step left in L2 (`config.l2`
says how this holds for the workload run).  `--graph` replays one CUDA graph
per step instead of calling the library each step.  `e2e` is the same metric through the
host-buffer entry point (pinned host memory, copies in and out inside the
timed region).  The reference arm (--impl reference) times the fp64 CPU
oracle on the host cores on bounded samples of the same workload.

Multi-GPU: the workload is a batch of independent sequences, so N ranks run N
independent replicas (one per GPU, weak scaling) with no collective on the
data path; only the timing uses a barrier and a max-reduction.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import mca_inputs  # noqa: E402

METRIC = "mixed-chunk attn fwd tokens/s and TFLOP/s at 1 GB300; % of bf16 tensor peak"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# ---------------------------------------------------------------- ranks
def rank_seed(seed: int, rank: int) -> int:
    """Input seed of one rank: every rank runs its own independent problem
    (another batch of sequences); rank 0 keeps the workload's own seed."""
    return seed + 1000 * rank


def reduce_max(x: float, device) -> float:
    """Max of `x` over the ranks of the default process group (x itself
    without one): the job's time is its slowest rank's."""
    dist = torch.distributed
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    tt = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def barrier():
    dist = torch.distributed
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


def whole_job_rate(world: int, units_per_rank_step: float, steps: int, max_seconds: float) -> float:
    """Units per second of the whole job: every rank processed its own
    units_per_rank_step each step, over the slowest rank's time."""
    return world * units_per_rank_step * steps / max_seconds


# ---------------------------------------------------------------- work accounting
def algorithmic_flops(w, lin_norm: int = 0) -> float:
    """Per forward pass: per chunk 2*P*(s+e) for the intra-chunk scores and
    relu^2-weighted values over the P unmasked (query, key) pairs, plus
    4*C*s*e for the chunk state and the global term (none without a global
    term)."""
    P = w.C * (w.C + 1) // 2 if w.causal else w.C * w.C
    per_chunk = 2.0 * P * (w.s + w.e) + (0.0 if lin_norm == 3 else 4.0 * w.C * w.s * w.e)
    return per_chunk * w.B * w.G


def algorithmic_bytes(w) -> float:
    """Compulsory HBM traffic of one pass: read Z, V, U once, write O once."""
    es = 2 if w.dtype == "bf16" else 4
    return float(w.B * w.n * (w.s + 3 * w.e) * es)


def kernel_algorithmic_bytes(w, kernel: str) -> float:
    """Compulsory HBM bytes of one launch of a forward kernel: what it must
    read of Z, V, U and write of O (its intermediates excluded).  The walkers
    read Z and V; the output kernels (row-pair, fused, and the one reading
    stored relu^2 weights) read V and U and write O; the T-row kernel and the
    relu^2-weight kernel read Z."""
    es = 2 if w.dtype == "bf16" else 4
    tokens = w.B * w.n
    if kernel == "tc_chunk_walk":
        return float(tokens * (w.s + w.e) * es)
    if kernel in ("tc_chunk_pair", "tc_chunk_fused", "tc_chunk_attn"):
        return float(tokens * 3 * w.e * es)
    if kernel in ("tc_affine_rows", "tc_chunk_prep"):
        return float(tokens * w.s * es)
    if kernel == "tc_seg_carry":
        return 0.0
    return algorithmic_bytes(w)  # the CUDA-core kernels: the whole pass


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(PEAKS_FALLBACK), "fallback"


FORWARD_KERNEL_SOURCES = ("tc.cu", "tc_common.cuh", "tc_prep.cuh", "tc_attn.cuh", "tc_fused.cuh",
                          "tc_walk.cuh", "tc_pair.cuh", "ptx.cuh")


def kernel_source_sha() -> str:
    """Hash of the sources of the tensor-core forward kernels and their launch."""
    csrc = os.path.join(ROOT, "flash_mixed_chunk_gb300", "csrc")
    h = hashlib.sha256()
    for f in FORWARD_KERNEL_SOURCES:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    sha = kernel_source_sha()
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        kv = dict(tok.split("=", 1) for tok in line.split() if "=" in tok)
        if (kv.get("kernel") == kernel and kv.get("workload") == workload
                and kv.get("source_sha") == sha):
            return float(kv["dram_bytes_per_launch"])
    return None


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (every 50 ms) of SM clock and throttle reasons."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def wait_first(self, timeout_s: float = 5.0) -> bool:
        """Wait (bounded) until nvidia-smi has printed its first sample."""
        t_end = time.time() + timeout_s
        while self.proc is not None and not self.samples and time.time() < t_end:
            time.sleep(0.01)
        return bool(self.samples)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float, label: str = "timed"):
        rows = [s for t, s in self.samples if t0 <= t <= t1]
        window = label
        if not rows:  # timed region shorter than the sampling period
            near = sorted(self.samples, key=lambda ts: min(abs(ts[0] - t0), abs(ts[0] - t1)))
            rows = [s for _, s in near[:2]]
            window = "nearest"
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm), "window": window}


# ---------------------------------------------------------------- CPU oracle timing
def oracle_sample_rate(w, inputs64, gamma, beta, budget_s: float):
    """Time the oracle on a bounded sample of the workload: the outputs of the
    first m chunks of batch element 0 (in causal mode they need only chunks
    < m; otherwise all chunks), with m grown up to the whole sequence, then the
    whole workload (every batch element) repeated, until one measurement takes
    about `budget_s`.  Returns (tokens/s, seconds, description, threads)."""
    import oracle
    Z, V, U = inputs64
    m = 1
    while True:
        rows = np.arange(m * w.C, dtype=np.int64)
        t = time.perf_counter()
        oracle.rows(Z, V, U, gamma, beta, w.C, w.causal, rows)
        dt = time.perf_counter() - t
        if dt >= budget_s:
            return m * w.C / dt, dt, f"outputs of the first {m} chunk(s) of batch element 0", \
                oracle.max_threads()
        if m >= w.G:
            break
        m = min(w.G, max(m + 1, int(m * budget_s / max(dt, 1e-3))))
    reps = 0
    t = time.perf_counter()
    while True:
        oracle.forward(Z, V, U, gamma, beta, w.C, w.causal)
        reps += 1
        dt = time.perf_counter() - t
        if dt >= budget_s:
            break
    return reps * w.B * w.n / dt, dt, f"{reps} full forward pass(es) of all {w.B} batch " \
        "element(s)", oracle.max_threads()


def host_cores() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def run_reference(args, w):
    """Reference arm: the fp64 CPU oracle as it stands, on host cores.  It
    runs on rank 0 only, so it takes every core of the host, whatever thread
    count a launcher set for the ranks (torchrun sets one)."""
    import oracle
    oracle.build()
    threads = host_cores()
    seed = mca_inputs.WORKLOAD_ORDER.index(w.name) + 1
    Z, V, U, gamma, beta = mca_inputs.workload_inputs(w, seed)
    inputs64 = tuple(x.to(torch.float64).numpy() for x in (Z, V, U))
    g64, b64 = gamma.double().numpy(), beta.double().numpy()
    qs, ln = variant_of(args, w)
    variant = {} if qs is None and ln == 0 else {"quad_scale": qs, "lin_norm": ln}
    # size each step so that warm-up + steps stay within about two minutes
    per_step = max(0.05, min(20.0, 120.0 / max(1, args.steps + args.warmup)))
    # each step: the outputs of the first m chunks of batch element 0, m sized
    # so that one step takes about `per_step` seconds (at most the sequence)
    m = 1
    while True:
        rows = np.arange(m * w.C, dtype=np.int64)
        t = time.perf_counter()
        oracle.rows(*inputs64, g64, b64, w.C, w.causal, rows, nthreads=threads, **variant)
        dt = time.perf_counter() - t
        if dt >= per_step or m >= w.G:
            break
        m = min(w.G, max(m + 1, int(m * per_step / max(dt, 1e-3))))
    for _ in range(args.warmup):
        oracle.rows(*inputs64, g64, b64, w.C, w.causal, rows, nthreads=threads, **variant)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle.rows(*inputs64, g64, b64, w.C, w.causal, rows, nthreads=threads, **variant)
    dt = time.perf_counter() - t
    value = args.steps * m * w.C / dt
    sample = (f"outputs of the first {m} chunk(s) of batch element 0 of {w.name} per step "
              f"({m * w.C} tokens; fp64 oracle, OpenMP)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, args),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


LIN_NORMS = {"n": 0, "summed": 1, "position": 2, "none": 3}


def variant_of(args, w):
    """(quad_scale or None, lin_norm) from --quad-scale / --lin-norm; "cs" is
    the page's 1/(C s)."""
    qs = None
    if args.quad_scale is not None:
        qs = 1.0 / (w.C * w.s) if args.quad_scale == "cs" else float(args.quad_scale)
    return qs, LIN_NORMS[args.lin_norm or w.lin_norm]


L2_BYTES = 129 * 2 ** 20


def l2_note(w) -> str:
    """How the timed steps avoid L2 reuse between iterations, as it applies."""
    es = 2 if w.dtype == "bf16" else 4
    set_bytes = w.B * w.n * (w.s + 3 * w.e) * es
    if set_bytes > L2_BYTES:
        return "inputs larger than L2, 3 rotating buffer sets"
    if 3 * set_bytes > L2_BYTES:
        return (f"3 rotating buffer sets of {set_bytes / 2 ** 20:.1f} MB, together larger "
                "than L2")
    return (f"3 rotating buffer sets of {set_bytes / 2 ** 20:.2f} MB: L2-resident "
            "(a launch-bound shape)")


def config_of(w, args=None):
    return {"workload": w.name, "B": w.B, "n": w.n, "C": w.C, "G": w.G, "s": w.s, "e": w.e,
            "causal": w.causal, "io_dtype": w.dtype, "accumulate": "fp32",
            "l2": l2_note(w),
            **({} if args is None or not getattr(args, "graph", False)
               else {"launch": "CUDA graph replay, one graph per step"}),
            "parallelism": "replicas (one independent problem per GPU)",
            **({} if args is None or (args.quad_scale is None and
                                      (args.lin_norm or w.lin_norm) == "n") else
               {"quad_scale": variant_of(args, w)[0] or 1.0 / (w.C * w.C),
                "lin_norm": args.lin_norm or w.lin_norm})}


# ---------------------------------------------------------------- decode
def decode_bytes_per_token(s, e, C, i):
    """Bytes one bf16 decode step must move per sequence at chunk index i: the
    bf16 copy of the carried state (s x e), the i cached Z and V rows of its
    chunk, the token's z, v, u and its output o; plus, at the chunk's last
    token, the fold (cache read once, fp32 state read and written, bf16 copy
    written)."""
    b = 2 * s * e + 2 * i * (s + e) + 2 * (s + 3 * e)
    if i == C - 1:
        b += 2 * C * (s + e) + 10 * s * e
    return b


def run_decode(args, device):
    """Autoregressive decoding of B sequences in lockstep through
    flash_mca_decode_step: K consecutive positions from t0 (whole chunks, so
    every chunk index and one fold per chunk are in the timed region)."""
    import flash_mixed_chunk_gb300 as fm
    torch.cuda.set_device(device)
    B, s, e, C = args.decode_batch, 128, 1536, 256
    t0, K, W = 4 * C, 2 * C, C
    n_norm = 16 * C
    qs, ln = variant_of(args, mca_inputs.WORKLOADS["gau_base_causal"])
    g = torch.Generator().manual_seed(11)
    rows = W + K
    z = torch.nn.functional.silu(torch.randn(rows, B, s, generator=g)).to(torch.bfloat16).to(device)
    v = torch.nn.functional.silu(torch.randn(rows, B, e, generator=g)).to(torch.bfloat16).to(device)
    u = torch.nn.functional.silu(torch.randn(rows, B, e, generator=g)).to(torch.bfloat16).to(device)
    gamma = (1 + 0.1 * torch.randn(4, s, generator=g)).to(device)
    beta = (0.1 * torch.randn(4, s, generator=g)).to(device)
    o = torch.empty(B, e, dtype=torch.bfloat16, device=device)
    state = torch.empty(fm.flash_mca_decode_state_bytes(B, s, e, C, fm.FMCA_BF16),
                        dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    fm.flash_mca_decode_reset(state, B, s, e, C, fm.FMCA_BF16, stream)
    # positions t0 - W .. t0 - 1 warm up (the state then holds earlier chunks)
    for k in range(W):
        fm.flash_mca_decode_step(z[k], v[k], u[k], gamma, beta, o, C, t0 - W + k, state, n_norm,
                                 qs, ln, stream)
    torch.cuda.synchronize(device)
    sampler = ClockSampler(device.index or 0)
    sampler.start()
    sampler.wait_first()
    # the timed loop calls the C entry point directly (pointers prepared
    # above), so that it measures the library, not Python argument checks
    opts = fm.flash_mca_default_options(C)
    if qs is not None:
        opts.quad_scale = qs
    opts.lin_norm = ln
    import ctypes
    call = fm.lib.flash_mca_decode_step
    sp = stream.cuda_stream
    zp = [z[W + k].data_ptr() for k in range(K)]
    vp = [v[W + k].data_ptr() for k in range(K)]
    up = [u[W + k].data_ptr() for k in range(K)]
    gp, bp, op, stp, stb = gamma.data_ptr(), beta.data_ptr(), o.data_ptr(), state.data_ptr(), \
        state.numel()
    ob = ctypes.byref(opts)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    a.record(stream)
    h0 = time.perf_counter()
    for k in range(K):
        rc = call(zp[k], vp[k], up[k], gp, bp, op, B, s, e, C, t0 + k, n_norm, fm.FMCA_BF16, ob,
                  stp, stb, sp)
        if rc:
            raise RuntimeError(fm.flash_mca_status_string(rc))
    host_us = (time.perf_counter() - h0) / K * 1e6
    b.record(stream)
    torch.cuda.synchronize(device)
    wall1 = time.time()
    sampler.stop()
    st, where = fm.flash_mca_device_status()
    if st != fm.FMCA_OK:
        raise RuntimeError(f"device status {fm.flash_mca_status_string(st)} at {where}")
    ms = a.elapsed_time(b)
    nbytes = B * sum(decode_bytes_per_token(s, e, C, (t0 + k) % C) for k in range(K))
    peaks, peak_kind = load_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", PEAKS_FALLBACK["hbm_gbs"]))
    achieved = nbytes / (ms / 1e3) / 1e9
    folds = sum(1 for k in range(K) if (t0 + k) % C == C - 1)
    line = {
        "metric": "mixed-chunk attn decode tokens/s (B sequences in lockstep) at 1 GB300",
        "value": B * K / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": K, "warmup": W,
        "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "decode", "B": B, "s": s, "e": e, "C": C,
                   "positions": f"{t0}..{t0 + K - 1}", "n_norm": n_norm,
                   **({} if qs is None and ln == 0 else {"quad_scale": qs, "lin_norm": args.lin_norm})},
        "roofline": {"bound": "hbm", "kernel": "decode step (decode_token + decode_fold)",
                     "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": None,
                     "algorithmic_bytes_per_step": nbytes / K,
                     "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)"},
        "gpu_launches": K + folds,
        "host_enqueue_us_per_step": host_us,
        "clocks": sampler.summary(wall0, wall1),
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- backward
# fp32 CUDA-core rate of a GB300: 152 SMs x 128 FP32 lanes x 2 FLOP x 2.07 GHz
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def run_backward(args, w, device):
    """The backward pass through flash_mca_backward on the workload's shape:
    K steps of dZ, dV, dU, dgamma, dbeta for a fixed dO, inputs resident."""
    import flash_mixed_chunk_gb300 as fm
    torch.cuda.set_device(device)
    seed = mca_inputs.WORKLOAD_ORDER.index(w.name) + 1
    Z, V, U, gamma, beta = (t.to(device) for t in mca_inputs.workload_inputs(w, seed))
    dO = torch.randn(w.B, w.n, w.e, generator=torch.Generator().manual_seed(seed + 100)).to(
        Z.dtype).to(device)
    qs, ln = variant_of(args, w)
    dZ, dV, dU = torch.empty_like(Z), torch.empty_like(V), torch.empty_like(U)
    dg = torch.empty(4, w.s, device=device)
    db = torch.empty_like(dg)
    ws = torch.empty(fm.flash_mca_backward_workspace_bytes(w.B, w.n, w.s, w.e, w.C, w.causal,
                                                           fm.FMCA_BF16 if w.dtype == "bf16"
                                                           else fm.FMCA_F32),
                     dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    if args.saved:
        # the forward pass's intermediates, kept in the workspace for every step
        O = torch.empty_like(U)
        fm.flash_mca_forward_ex(Z, V, U, gamma, beta, O, w.C, w.causal, ws, qs, ln,
                                fm.FMCA_PATH_AUTO, stream)

    def step():
        fm.flash_mca_backward(Z, V, U, gamma, beta, dO, dZ, dV, dU, dg, db, w.C, w.causal, ws, qs,
                              ln, stream, saved=args.saved)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)
    sampler = ClockSampler(device.index or 0)
    sampler.start()
    sampler.wait_first()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    a.record(stream)
    for _ in range(args.steps):
        step()
    b.record(stream)
    torch.cuda.synchronize(device)
    wall1 = time.time()
    sampler.stop()
    st, where = fm.flash_mca_device_status()
    if st != fm.FMCA_OK:
        raise RuntimeError(f"device status {fm.flash_mca_status_string(st)} at {where}")
    ms = a.elapsed_time(b) / args.steps
    # the gradient's own products, twice the forward pass's (recompute not counted)
    flops = 2.0 * algorithmic_flops(w, ln)
    achieved = flops / (ms / 1e3) / 1e12
    dcode = fm.FMCA_BF16 if w.dtype == "bf16" else fm.FMCA_F32
    tc = fm.flash_mca_auto_path(w.B, w.n, w.s, w.e, w.C, w.causal, dcode) == fm.FMCA_PATH_TCGEN05
    if tc:
        peaks, peak_kind = load_peaks()
        peak = float(peaks.get("bf16_tflops", PEAKS_FALLBACK["bf16_tflops"]))
        roof = {"bound": "tensor", "kernel": "whole backward (tcgen05 products + elementwise)",
                "peak_source": f"bf16_tflops ({peak_kind})"}
        dtype = "bf16 (tensor cores, fp32 accumulate)"
    else:
        peak = FP32_ALU_TFLOPS
        roof = {"bound": "alu", "kernel": "whole backward (SIMT fp32)",
                "peak_source": "fp32 CUDA-core rate from unit counts and max clock"}
        dtype = "f32 (CUDA cores; I/O " + w.dtype + ")"
    roof.update({"achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                 "traffic": None, "algorithmic_flops_per_step": flops})
    line = {
        "metric": "mixed-chunk attn backward tokens/s at 1 GB300",
        "value": w.B * w.n / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": dtype, "data": "synthetic",
        "config": {**config_of(w, args),
                   "pass": "backward, forward intermediates kept" if args.saved else "backward"},
        "roofline": roof,
        "gpu_launches": args.steps * fm.flash_mca_backward_launch_count(
            w.B, w.n, w.s, w.e, w.C, w.causal, dcode, qs, ln, saved=args.saved),
        "clocks": sampler.summary(wall0, wall1),
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- projections
def run_projections(args, w, device):
    """The GAU projections around the core on the workload's token count:
    U, V, Z = SiLU(X [W_u|W_v|W_z]) and Out = Y W_o, d = e / 2, on the tensor
    cores; one JSON line per GEMM."""
    import flash_mixed_chunk_gb300 as fm
    torch.cuda.set_device(device)
    M, e, s = w.B * w.n, w.e, w.s
    d = e // 2
    g = torch.Generator().manual_seed(21)
    X = torch.randn(M, d, generator=g).to(torch.bfloat16).to(device)
    Wt = (d ** -0.5 * torch.randn(2 * e + s, d, generator=g)).to(torch.bfloat16).to(device)
    Y = torch.randn(M, e, generator=g).to(torch.bfloat16).to(device)
    Wo_t = (e ** -0.5 * torch.randn(d, e, generator=g)).to(torch.bfloat16).to(device)
    U = torch.empty(M, e, dtype=torch.bfloat16, device=device)
    V, Z = torch.empty_like(U), torch.empty(M, s, dtype=torch.bfloat16, device=device)
    Out = torch.empty(M, d, dtype=torch.bfloat16, device=device)
    stream = torch.cuda.current_stream(device)
    peaks, peak_kind = load_peaks()
    bf16_peak = float(peaks.get("bf16_tflops", PEAKS_FALLBACK["bf16_tflops"]))
    cases = [("project", lambda: fm.flash_mca_gau_project(X, Wt, U, V, Z, stream),
              2.0 * M * d * (2 * e + s), f"X[{M},{d}] x [W_u|W_v|W_z][{d},{2 * e + s}], SiLU"),
             ("output", lambda: fm.flash_mca_gau_output(Y, Wo_t, Out, stream),
              2.0 * M * e * d, f"Y[{M},{e}] x W_o[{e},{d}]")]
    for name, fn, flops, what in cases:
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize(device)
        sampler = ClockSampler(device.index or 0)
        sampler.start()
        sampler.wait_first()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        wall0 = time.time()
        a.record(stream)
        for _ in range(args.steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize(device)
        wall1 = time.time()
        sampler.stop()
        st, where = fm.flash_mca_device_status()
        if st != fm.FMCA_OK:
            raise RuntimeError(f"device status {fm.flash_mca_status_string(st)} at {where}")
        ms = a.elapsed_time(b) / args.steps
        tf = flops / (ms / 1e3) / 1e12
        print(json.dumps({
            "metric": f"GAU {name} projection TFLOP/s at 1 GB300", "value": tf, "unit": "TFLOP/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": {"workload": f"gau_{name}_{w.name}", "gemm": what},
            "roofline": {"bound": "tensor", "kernel": "tc_gemm", "achieved": tf,
                         "peak": bf16_peak, "unit": "TFLOP/s", "frac": tf / bf16_peak,
                         "traffic": None,
                         "peak_source": f"{peak_kind} bf16_tflops (MEASURED_PEAKS.json)"},
            "gpu_launches": args.steps, "clocks": sampler.summary(wall0, wall1)}), flush=True)


# ---------------------------------------------------------------- our arm
def run_ours(args, w, rank, world, device):
    import flash_mixed_chunk_gb300 as fm

    torch.cuda.set_device(device)
    seed = rank_seed(mca_inputs.WORKLOAD_ORDER.index(w.name) + 1, rank)
    Zc, Vc, Uc, gc, bc = mca_inputs.workload_inputs(w, seed)
    dt_code = fm.FMCA_BF16 if w.dtype == "bf16" else fm.FMCA_F32
    path = fm.flash_mca_auto_path(w.B, w.n, w.s, w.e, w.C, w.causal, dt_code)
    quad_scale, lin_norm = variant_of(args, w)
    nl = fm.flash_mca_launch_count(w.B, w.n, w.s, w.e, w.C, w.causal, dt_code,
                                   quad_scale=quad_scale, lin_norm=lin_norm)
    sets = []
    for _ in range(3):
        sets.append(dict(Z=Zc.to(device), V=Vc.to(device), U=Uc.to(device),
                         O=torch.empty((w.B, w.n, w.e), dtype=Zc.dtype, device=device)))
    gd, bd = gc.to(device), bc.to(device)
    ws = torch.empty(fm.flash_mca_workspace_bytes(w.B, w.n, w.s, w.e, w.C, w.causal, dt_code),
                     dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    def step(i, events=None):
        s = sets[i % 3]
        if events is None and (quad_scale is not None or lin_norm):
            fm.flash_mca_forward_ex(s["Z"], s["V"], s["U"], gd, bd, s["O"], w.C, w.causal, ws,
                                    quad_scale, lin_norm, fm.FMCA_PATH_AUTO, stream)
        elif events is None:
            fm.flash_mca_forward(s["Z"], s["V"], s["U"], gd, bd, s["O"], w.C, w.causal, ws, stream)
        else:
            fm.flash_mca_forward_timed(s["Z"], s["V"], s["U"], gd, bd, s["O"], w.C, w.causal, ws,
                                       events, fm.FMCA_PATH_AUTO, stream, quad_scale, lin_norm)

    sampler = ClockSampler(torch.cuda.current_device() if device.index is None else device.index)
    sampler.start()
    sampler.wait_first()  # so that the run's window holds samples however short it is
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(device)
    st, where = fm.flash_mca_device_status()
    if st != fm.FMCA_OK:
        raise RuntimeError(f"device status {fm.flash_mca_status_string(st)} at {where}")

    graphs = None
    if args.graph:
        # one CUDA graph per buffer set, each holding one whole forward step
        # (its kernels and their programmatic dependencies); replayed in turn
        graphs = []
        for i in range(3):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                cap = torch.cuda.current_stream(device)
                si = sets[i]
                fm.flash_mca_forward_ex(si["Z"], si["V"], si["U"], gd, bd, si["O"], w.C,
                                        w.causal, ws, quad_scale, lin_norm, fm.FMCA_PATH_AUTO, cap)
            graphs.append(g)
        for i in range(args.warmup):
            graphs[i % 3].replay()
        torch.cuda.synchronize(device)

    # ---- timed region: exactly K steps of the forward pass, nothing between
    # its kernels (the library chains them with programmatic dependent launch)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(device)
    wall0 = time.time()
    t_start.record(stream)
    if graphs is not None:
        for i in range(args.steps):
            graphs[i % 3].replay()
    else:
        for i in range(args.steps):
            step(i)
    t_end.record(stream)
    torch.cuda.synchronize(device)
    wall1 = time.time()
    barrier()
    st, where = fm.flash_mca_device_status()
    if st != fm.FMCA_OK:
        raise RuntimeError(f"device status {fm.flash_mca_status_string(st)} at {where}")
    ms = reduce_max(t_start.elapsed_time(t_end), device)

    # ---- second timed pass of K steps with CUDA events recorded by the library
    # before the first kernel and after each kernel (on the launching stream):
    # the per-kernel split and the dominant kernel's duration for the roofline
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(nl + 1)]
              for _ in range(args.steps)]
    for evs in events:  # create the CUDA event handles outside the timed pass
        for ev in evs:
            ev.record(stream)
    torch.cuda.synchronize(device)
    k_start = torch.cuda.Event(enable_timing=True)
    k_end = torch.cuda.Event(enable_timing=True)
    k_start.record(stream)
    for i in range(args.steps):
        step(i, events[i])
    k_end.record(stream)
    torch.cuda.synchronize(device)
    ms_events = k_start.elapsed_time(k_end)
    per_kernel_ms = [statistics.fmean(ev[k].elapsed_time(ev[k + 1]) for ev in events)
                     for k in range(nl)]
    step_us = sorted(1e3 * ev[0].elapsed_time(ev[nl]) for ev in events)

    # ---- end to end through the host-buffer entry point
    pin = [t.pin_memory() for t in (Zc, Vc, Uc, gc, bc)]
    Oh = torch.empty((w.B, w.n, w.e), dtype=Zc.dtype).pin_memory()
    arena = torch.empty(fm.flash_mca_host_arena_bytes(w.B, w.n, w.s, w.e, w.C, w.causal, dt_code),
                        dtype=torch.uint8, device=device)
    k_e2e = max(3, min(args.steps, 200))
    for _ in range(3):
        fm.flash_mca_forward_host(*pin, Oh, w.C, w.causal, arena, stream)
    barrier()
    t = time.perf_counter()
    for _ in range(k_e2e):
        fm.flash_mca_forward_host(*pin, Oh, w.C, w.causal, arena, stream)
    e2e_s = reduce_max(time.perf_counter() - t, device)
    wall2 = time.time()
    sampler.stop()
    h2d = sum(t.numel() * t.element_size() for t in pin)
    d2h = Oh.numel() * Oh.element_size()

    if rank != 0:
        return
    peaks, peak_kind = load_peaks()
    tokens = w.B * w.n
    value = whole_job_rate(world, tokens, args.steps, ms / 1e3)
    flops = algorithmic_flops(w, lin_norm)
    tflops = world * flops * args.steps / (ms / 1e3) / 1e12
    if path != fm.FMCA_PATH_TCGEN05:
        kernel_names = ["simt_chunk_state", "simt_chunk_scan", "simt_chunk_output"]
    elif lin_norm == fm.FMCA_LIN_NORM_NONE:
        # chunks of up to 256 tokens: the T0 / T1 rows, then the fused kernel;
        # longer (the quadratic-only model): the relu^2 weights through HBM
        kernel_names = (["tc_affine_rows", "tc_chunk_fused"] if w.C <= 256
                        else ["tc_chunk_prep", "tc_chunk_attn"])
    else:
        # the segment walkers, the carries (with more than one segment or
        # bidirectional), the output kernel (both row tiles of a chunk of 256
        # per unit, else one)
        out_kernel = "tc_chunk_pair" if w.C == 256 else "tc_chunk_fused"
        kernel_names = (["tc_chunk_walk", out_kernel] if nl == 2
                        else ["tc_chunk_walk", "tc_seg_carry", out_kernel])
    kernels = {name: {"ms": per_kernel_ms[i], "share": per_kernel_ms[i] / sum(per_kernel_ms)}
               for i, name in enumerate(kernel_names)}
    dom = max(kernels, key=lambda k: kernels[k]["ms"])
    dom_ms = kernels[dom]["ms"]
    dom_bytes = kernel_algorithmic_bytes(w, dom)
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9
    hbm_peak = float(peaks.get("hbm_gbs", PEAKS_FALLBACK["hbm_gbs"]))
    bf16_peak = float(peaks.get("bf16_tflops", PEAKS_FALLBACK["bf16_tflops"]))
    traffic = profiled_traffic(dom, w.name)
    # the whole step: the pass's compulsory bytes over the step time, and the
    # profiled DRAM bytes of all its launches (null unless every kernel of the
    # step was profiled on the current sources)
    step_gbs = algorithmic_bytes(w) / (ms / args.steps / 1e3) / 1e9
    per_kernel_traffic = [profiled_traffic(k, w.name) for k in kernel_names]
    step_traffic = (sum(per_kernel_traffic)
                    if per_kernel_traffic and all(t is not None for t in per_kernel_traffic)
                    else None)

    # ---- CPU baseline: the oracle as it stands, bounded sample, host cores
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        inputs64 = tuple(x.to(torch.float64).numpy() for x in (Zc, Vc, Uc))
        rate, dt, what, threads = oracle_sample_rate(w, inputs64, gc.double().numpy(),
                                                     bc.double().numpy(), args.cpu_budget)
        cpu = {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"{what} of {w.name} ({dt:.1f} s; fp64 oracle, OpenMP)"}

    # clocks over the timed pass, the per-kernel event pass and the host-buffer
    # pass (all of them keep the GPU busy); the sampler was started, and its
    # first sample awaited, before the warm-up
    clocks = sampler.summary(wall0, wall2, "timed+events+e2e")
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": config_of(w, args),
        "tflops": tflops, "pct_bf16_peak": 100.0 * tflops / bf16_peak,
        "hbm_gbs_step": world * algorithmic_bytes(w) * args.steps / (ms / 1e3) / 1e9,
        "path": "tcgen05" if path == fm.FMCA_PATH_TCGEN05 else "simt",
        "kernels": kernels,
        "ms_per_step_with_kernel_events": ms_events / args.steps,
        "step_us_spread": {"min": step_us[0], "median": statistics.median(step_us),
                           "max": step_us[-1], "pass": "per-kernel event pass"},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm_peak,
                     "unit": "GB/s", "frac": achieved / hbm_peak, "traffic": traffic,
                     "algorithmic_bytes_per_launch": dom_bytes,
                     "step_achieved": step_gbs, "step_frac": step_gbs / hbm_peak,
                     "step_algorithmic_bytes": algorithmic_bytes(w),
                     "step_traffic": step_traffic,
                     "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s"},
        "cpu_baseline": cpu,
        "e2e": {"value": whole_job_rate(world, tokens, k_e2e, e2e_s), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": k_e2e},
        "gpu_launches": nl * args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long_causal", choices=list(mca_inputs.WORKLOADS))
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle work for the CPU baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quad-scale", default=None,
                    help="intra-chunk weight scale: a number, or 'cs' for the page's 1/(C s) "
                         "(default: 1/C^2); the headline loop then runs flash_mca_forward_ex")
    ap.add_argument("--decode", action="store_true",
                    help="time the autoregressive decode step instead of the forward pass "
                         "(its own JSON line)")
    ap.add_argument("--decode-batch", type=int, default=8)
    ap.add_argument("--projections", action="store_true",
                    help="time the GAU projection GEMMs (tensor cores) on the workload's tokens")
    ap.add_argument("--saved", action="store_true",
                    help="with --backward: flash_mca_backward_saved (forward intermediates kept)")
    ap.add_argument("--graph", action="store_true",
                    help="time the forward steps as CUDA graph replays (one graph per step)")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward pass on the workload (its own JSON line)")
    ap.add_argument("--lin-norm", default=None, choices=list(LIN_NORMS),
                    help="global-term divisor: n, summed (tokens the sum covers), position "
                         "(t+1), or none (no global term; with C = n: FLASH-Quad); default: "
                         "the workload's (n for all but flash_quad_base)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    w = mca_inputs.WORKLOADS[args.workload]

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.decode:
        if rank == 0 and args.impl == "ours":
            run_decode(args, torch.device("cuda", local))
        return
    if args.backward:
        if rank == 0 and args.impl == "ours":
            run_backward(args, w, torch.device("cuda", local))
        return
    if args.projections:
        if rank == 0 and args.impl == "ours":
            run_projections(args, w, torch.device("cuda", local))
        return
    if args.impl == "reference":
        if rank == 0:
            run_reference(args, w)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl")
    device = torch.device("cuda", local)
    try:
        run_ours(args, w, rank, world, device)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
