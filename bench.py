#!/usr/bin/env python
"""Benchmark of the chunkwise KDA forward pass (tokens/s and % of the HBM roofline).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one call of the library's forward entry point over one batch of the
B=2, T=8192, H=32, d_k=d_v=128, C=64 bf16 per-channel-gate workload with an initial
state and the final state written. Inputs live in HBM before the timed region (816 MB
per step, larger than the 129 MB L2, so no flush is needed between steps). Rank 0
prints one JSON line. Under torchrun every rank runs its own batch (weak scaling; the
(sequence, head) units are independent, so ranks exchange nothing but the timing).

``--impl reference`` times the fp64 CPU oracle as it stands on this host's cores, each
step a bounded sample of (sequence, head) units of the same workload.
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import statistics
import os
import re
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "kda_b2_t8192_h32_d128_bf16"
METRIC = "chunk KDA fwd tokens/s at T=8192,H=32,d=128 bf16; % of roofline"
NOMINAL_HBM_GBS = 8000.0  # the nominal HBM3e bandwidth the roofline target is stated against


def metric_name(entry: str, workload: str) -> str:
    """The headline metric for the default run; otherwise one that names what was timed."""
    if entry == "chunk" and workload == WORKLOAD:
        return METRIC
    what = {"chunk": "chunk KDA fwd", "recurrent": "KDA recurrent decode step",
            "backward": "chunk KDA bwd (dq, dk, dv, dg, dbeta, dh0)"}[entry]
    return f"{what} tokens/s on {workload}"

# DRAM traffic per launch of the forward kernel, from an ncu capture of this workload
# (dram__bytes_read.sum + dram__bytes_write.sum), keyed by a hash of the code of the kernel
# it was taken on (comments ignored); any change to the code makes the figure stale
# (reported as null).
MEASURED_TRAFFIC = {
    # profiles/kda_fwd_pc_b2_t8192_h32_d128.md: 397.7 MB on the same 64 units over half the
    # tokens (B=2, T=4096), scaled by 2 to this workload
    ("kda_b2_t8192_h32_d128_bf16", "8e9d471b383ffba9"): 795_367_936,
}

# The translation unit of each forward kernel and the headers it includes.
KERNEL_SOURCES = {
    "kda_fwd_pc_kernel": ("kda_fwd_pc.cu", "kda_common.cuh", "tc_util.cuh", "tc5.cuh"),
    "kda_fwd_tc_kernel": ("kda_fwd_tc.cu", "kda_common.cuh", "tc_util.cuh", "tc5.cuh"),
    "kda_fwd_bf16_kernel": ("kda_fwd_bf16.cu", "kda_common.cuh"),
    "kda_fwd_f32_kernel": ("kda_fwd_f32.cu", "kda_common.cuh"),
    "kda_recurrent_kernel": ("kda_recurrent.cu", "kda_common.cuh"),
}


def _code_only(text: str) -> str:
    """The source without comments and with whitespace collapsed (string and character
    literals kept as they are), so that edits to comments leave the hash unchanged."""
    tok = re.compile(r'"(?:\\.|[^"\\])*"|\'(?:\\.|[^\'\\])*\'|//[^\n]*|/\*.*?\*/', re.S)
    text = tok.sub(lambda m: m.group(0) if m.group(0)[0] in "\"'" else " ", text)
    return " ".join(text.split())


def kernel_source_hash(kernel: str = "kda_fwd_pc_kernel") -> str:
    """Hash of the code (comments and layout ignored) of a kernel's translation unit and
    the headers it includes."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "chunkwise_gated_linear_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def algorithmic_bytes(x) -> int:
    """HBM bytes the method must move: q, k once per key head; v, o, g, beta (if any) per
    value head; h0 and ht once per (sequence, value head)."""
    e = 2 if x.dtype == "bf16" else 4
    T = x.T_total
    gate = 4 * x.d_k if x.gate == "channel" else 4
    per_tok = x.H_k * 2 * x.d_k * e + x.H_v * (2 * x.d_v * e + gate + (4 if x.beta is not None else 0))
    state = x.N * x.H_v * 4 * x.d_k * x.d_v * ((x.h0 is not None) + 1)
    # the front-end's per-head parameters (A_log, dt_bias), when present
    params = 0
    if getattr(x, "A_log", None) is not None:
        params = 4 * x.A_log.size + (4 * x.dt_bias.size if x.dt_bias is not None else 0)
    return T * per_tok + state + params


def backward_bytes(x) -> int:
    """HBM bytes the backward must move: the forward inputs (q, k, v, g, beta, h0), dO and
    dht in; dq, dk, dv, dg, dbeta and dh0 out."""
    e = 2 if x.dtype == "bf16" else 4
    gate = 4 * x.d_k if x.gate == "channel" else 4
    bet = 8 if x.beta is not None else 0  # beta in, dbeta out
    per_tok = x.H_k * 4 * x.d_k * e + x.H_v * (3 * x.d_v * e + 2 * gate + bet)
    state = x.N * x.H_v * 4 * x.d_k * x.d_v * ((x.h0 is not None) + 2)  # h0, dht, dh0
    return x.T_total * per_tok + state


def backward_flops(x, C=64) -> int:
    """Useful FLOPs of the backward's contractions as this library runs them, per (chunk,
    value head): the recomputed chunk factors (Gram, Aqk, U, W), the forward state scan
    (W S, Kb^T Vt), the adjoint scan (A^T dO, Kb dS, Qp^T dO, W^T dVt) and the gradients
    (dO S^T, dO Vt^T, dA Km, Vt dS^T, dVt S^T, dW Kp^T, dVt V^T, T^T dW, T^T dVt, dT T^T,
    T^T X, dM Km, dM^T Kp, dA^T Qp), masks not exploited; a tail chunk counts in full."""
    K, V = x.d_k, x.d_v
    mac = (3 * C * C * K + C * C * V                      # prep: Gram, Aqk, W, U
           + 2 * C * K * V                                # forward state scan
           + C * C * V + 3 * C * K * V                    # adjoint scan
           + 3 * C * K * V + 3 * C * C * V + 6 * C * C * K + 2 * C * C * C)  # gradients
    lens = x.lengths()
    chunks = int(sum((int(n) + C - 1) // C for n in lens))
    return 2 * mac * chunks * x.H_v


def algorithmic_flops(x, C=64) -> int:
    """Useful FLOPs of the chunk algorithm (causal halves counted once), per token and
    value head: Gram (strict lower) + Aqk (lower) + forward substitution on [Kp | V]
    + W S + Qp S + Aqk Vt + Kbar^T Vt."""
    dk, dv = x.d_k, x.d_v
    lo, lo_d = C * (C - 1) // 2, C * (C + 1) // 2
    per_chunk = 2 * (lo * dk + lo_d * dk + lo * (dk + dv) + 3 * C * dk * dv + lo_d * dv)
    return int(round(per_chunk / C * x.T_total * x.H_v))


def forward_kernel(x, sms: int) -> str:
    """The kernel the library's dispatch runs for this workload (see kda_api.cu): with
    d_k = d_v = 128 in bf16 the persistent producer/consumer kernel when the (sequence,
    head) units are at most 76 and at most half the SMs, else one CTA per unit."""
    units = x.N * x.H_v
    if x.dtype == "f32":
        return "kda_fwd_f32_kernel"
    if x.d_k == 128 and x.d_v == 128:
        return "kda_fwd_pc_kernel" if units <= 76 and 2 * units <= sms else "kda_fwd_tc_kernel"
    return "kda_fwd_bf16_kernel"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples taken during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for nm, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.path)
        sm.sort()
        med = sm[len(sm) // 2] if sm else None
        return {"sm_mhz": med, "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, value: float) -> float:
    if pg is None:
        return value
    import torch

    dev = "cuda" if torch.cuda.is_available() and pg.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def oracle_sample(x, n_units, threads=0):
    """Time the fp64 oracle on the first n_units (sequence, head) units; returns
    (seconds, equivalent tokens, threads used)."""
    from oracle import kda_fused_recurrence, kda_recurrence, oracle_threads

    units = [(n, h) for n in range(x.N) for h in range(x.H_v)][:n_units]
    t0 = time.perf_counter()
    if getattr(x, "meta", {}).get("frontend"):
        kda_fused_recurrence(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, x.scale,
                             qk_l2norm=x.qk_l2norm, beta_sigmoid=x.beta_sigmoid, A_log=x.A_log,
                             dt_bias=x.dt_bias, units=units, threads=threads)
    else:
        kda_recurrence(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, x.scale, units=units, threads=threads)
    dt = time.perf_counter() - t0
    lens = x.lengths()
    unit_tokens = sum(int(lens[n]) for n, _ in units)
    used = min(threads if threads > 0 else oracle_threads(), len(units))
    return dt, unit_tokens / x.H_v, used


def oracle_bwd_sample(x, do, dht, n_units, threads=0):
    """Time the fp64 backward oracle on the first n_units (sequence, head) units; returns
    (seconds, equivalent tokens, threads used)."""
    from oracle import kda_recurrence_bwd, oracle_threads

    units = [(n, h) for n in range(x.N) for h in range(x.H_v)][:n_units]
    t0 = time.perf_counter()
    kda_recurrence_bwd(x.q, x.k, x.v, x.g, x.beta, x.h0, do, dht, x.cu_seqlens, x.scale, units=units,
                       threads=threads)
    dt = time.perf_counter() - t0
    lens = x.lengths()
    unit_tokens = sum(int(lens[n]) for n, _ in units)
    used = min(threads if threads > 0 else oracle_threads(), len(units))
    return dt, unit_tokens / x.H_v, used


def run_reference(args, world, rank, pg):
    """--impl reference: the oracle as it stands, on the host cores, bounded samples (the
    token recurrence, or its reverse-mode gradients with --entry backward)."""
    import numpy as np

    from inputs import workload_inputs
    from oracle import oracle_threads

    if rank != 0:
        return
    x = workload_inputs(args.workload)
    n_units = max(1, min(oracle_threads(), x.N * x.H_v))
    entry = getattr(args, "entry", "chunk")
    backward = entry == "backward"
    if backward:
        # the cotangents of the backward benchmark (seeded as there)
        rng = np.random.default_rng(2000)
        do = rng.standard_normal(x.v.shape, dtype=np.float32)
        dht = rng.standard_normal((x.N, x.H_v, x.d_k, x.d_v), dtype=np.float32)
        sample_fn = lambda: oracle_bwd_sample(x, do, dht, n_units)  # noqa: E731
        what = "fp64 reverse-mode gradients of the token recurrence"
    else:
        sample_fn = lambda: oracle_sample(x, n_units)  # noqa: E731
        what = "fp64 token recurrence"
    for _ in range(args.warmup):
        sample_fn()
    tot_t, tot_tok, used = 0.0, 0.0, 1
    for _ in range(args.steps):
        dt, tok, used = sample_fn()
        tot_t += dt
        tot_tok += tok
    value = tot_tok / tot_t
    sample = (f"{n_units} of {x.N * x.H_v} (sequence, head) units of {args.workload} per step "
              f"({x.lengths()[0]} tokens each), {what}")
    line = {
        "impl": "reference", "metric": metric_name(entry, args.workload),
        "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * tot_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": args.workload, "sample": sample},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": used, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


E2E_H2D_STREAMS = 1


def run_ours(args, world, rank, local, pg):
    import numpy as np
    import torch

    from chunkwise_gated_linear_gb300 import kda
    from inputs import workload_frontend_inputs, workload_inputs

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lib = kda.lib()

    fe_on = args.frontend != "none"
    if fe_on:
        x = workload_frontend_inputs(args.workload, seed=1000 + rank)
    else:
        x = workload_inputs(args.workload, seed=1000 + rank)
    B = x.N                       # sequences
    Bp = 1 if x.varlen else B     # physical batch (packed sequences: one row of T_total tokens)
    T = x.T_total // Bp
    dt_io = torch.bfloat16 if x.dtype == "bf16" else torch.float32

    def host(a, dtype, shape):
        return torch.from_numpy(np.ascontiguousarray(a)).reshape(shape).to(dtype).pin_memory()

    gshape = (Bp, T, x.H_v, x.d_k) if x.gate == "channel" else (Bp, T, x.H_v)
    H = {
        "q": host(x.q, dt_io, (Bp, T, x.H_k, x.d_k)), "k": host(x.k, dt_io, (Bp, T, x.H_k, x.d_k)),
        "v": host(x.v, dt_io, (Bp, T, x.H_v, x.d_v)), "g": host(x.g, torch.float32, gshape),
    }
    if x.beta is not None:  # no beta: the decay-only recurrence
        H["beta"] = host(x.beta, torch.float32, (Bp, T, x.H_v))
    if x.h0 is not None:  # no h0: a zero initial state
        H["h0"] = host(x.h0, torch.float32, (B, x.H_v, x.d_k, x.d_v))
    if fe_on:  # the gate's per-head parameters
        H["A_log"] = host(x.A_log, torch.float32, (x.H_v,))
        H["dt_bias"] = host(x.dt_bias, torch.float32, x.dt_bias.shape)
    inputs = [key for key in ("q", "k", "v", "g", "beta", "h0", "A_log", "dt_bias") if key in H]
    D = {key: t.to(dev) for key, t in H.items()}
    D["o"] = torch.empty((Bp, T, x.H_v, x.d_v), dtype=dt_io, device=dev)
    D["ht"] = torch.empty((B, x.H_v, x.d_k, x.d_v), dtype=torch.float32, device=dev)
    H["o"] = torch.empty_like(D["o"], device="cpu").pin_memory()
    H["ht"] = torch.empty_like(D["ht"], device="cpu").pin_memory()
    cu = torch.from_numpy(x.cu_seqlens.astype(np.int32)).to(dev) if x.varlen else None
    stream = torch.cuda.Stream(device=dev)
    sh = stream.cuda_stream
    plain_call = args.entry == "chunk" and x.dtype == "bf16" and x.gate == "channel" and not fe_on

    def make_call(Ds):
        """One library call on the device buffers Ds, on `stream`."""
        ptr = lambda key: Ds[key].data_ptr() if key in Ds else None  # noqa: E731
        params = kda.kda_fwd_params(
            ptr("q"), ptr("k"), ptr("v"), ptr("g"), ptr("beta"), ptr("h0"), ptr("o"), ptr("ht"), B, T, x.H_k,
            x.H_v, x.d_k, x.d_v, 64, x.scale, None if cu is None else cu.data_ptr(),
            kda.KDA_DTYPE_BF16 if x.dtype == "bf16" else kda.KDA_DTYPE_F32,
            kda.KDA_GATE_PER_CHANNEL if x.gate == "channel" else kda.KDA_GATE_PER_HEAD,
            kda.KDA_FLAG_UNFUSED_FRONTEND if args.frontend == "unfused" else 0)
        fe = kda.kda_frontend(1, 1 if x.beta is not None else 0, ptr("A_log"), ptr("dt_bias")) if fe_on else None

        def call():
            # kda_chunk_fwd (the plain argument-list entry point) when the workload fits its
            # argument list, else the struct entry points of the same ABI
            if fe_on:
                fn = lib.kda_recurrent_fwd_fused if args.entry == "recurrent" else lib.kda_chunk_fwd_fused
                st = fn(ctypes.byref(params), ctypes.byref(fe), sh)
            elif plain_call:
                st = lib.kda_chunk_fwd(ptr("q"), ptr("k"), ptr("v"), ptr("g"), ptr("beta"), ptr("h0"), ptr("o"),
                                       ptr("ht"), B, T, x.H_k, x.H_v, x.d_k, x.d_v, 64, x.scale,
                                       None if cu is None else cu.data_ptr(), sh)
            elif args.entry == "recurrent":
                st = lib.kda_recurrent_fwd_ex(ctypes.byref(params), sh)
            else:
                st = lib.kda_chunk_fwd_ex(ctypes.byref(params), sh)
            if st != 0:
                raise RuntimeError(kda.status_string(st))
        return call

    call = make_call(D)

    # End to end: every step copies its inputs from pinned host memory and reads its results
    # back. Steps are double-buffered over two sets of device buffers, with one copy stream
    # per direction, so that step i + 1's inputs travel while step i computes and step i - 1's
    # results come back (as a serving loop would run it).
    D2 = {key: torch.empty_like(D[key]) for key in inputs + ["o", "ht"]}
    sets = [D, D2]
    calls = [call, make_call(D2)]
    s_out = torch.cuda.Stream(device=dev)
    # input copy streams (more than one measured no faster: the host link is saturated)
    s_ins = [torch.cuda.Stream(device=dev) for _ in range(E2E_H2D_STREAMS)]
    s_in = s_ins[0]
    ev_in = [[torch.cuda.Event() for _ in range(E2E_H2D_STREAMS)] for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    step_no = [0]

    def e2e_step():
        i = step_no[0]
        step_no[0] += 1
        j = i & 1
        Dj = sets[j]
        for si, st_in in enumerate(s_ins):
            with torch.cuda.stream(st_in):
                if i >= 2:
                    st_in.wait_event(ev_done[j])  # step i - 2 has read set j's inputs
                for key in inputs[si::E2E_H2D_STREAMS]:
                    Dj[key].copy_(H[key], non_blocking=True)
                ev_in[j][si].record(st_in)
        for ev in ev_in[j]:
            stream.wait_event(ev)
        if i >= 2:
            stream.wait_event(ev_out[j])  # step i - 2's results in set j have been read back
        calls[j]()
        ev_done[j].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[j])
            H["o"].copy_(Dj["o"], non_blocking=True)
            H["ht"].copy_(Dj["ht"], non_blocking=True)
            ev_out[j].record(s_out)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize(dev)

    # device-resident throughput: exactly K launches, CUDA events on the launch stream
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev_step = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    with ClockSampler(local) as clk:
        barrier(pg)
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        for i in range(args.steps):
            ev_step[i].record(stream)
            call()
        ev_step[args.steps].record(stream)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(pg)
    ms = ev0.elapsed_time(ev1) / args.steps
    ms_median = statistics.median(ev_step[i].elapsed_time(ev_step[i + 1]) for i in range(args.steps))
    clocks = clk.summary()
    ms_max = max_over_ranks(pg, ms)
    tokens = x.T_total
    value = tokens * world / (ms_max / 1000.0)

    # end to end through the C ABI with host buffers: H2D inputs, call, D2H results
    for _ in range(max(2, args.warmup // 2)):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(pg)
    ev2, ev3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step_no[0] = 0  # the timed steps start with empty pipelines
    ev2.record(s_in)
    for st_in in s_ins[1:]:
        st_in.wait_stream(s_in)
    for _ in range(args.steps):
        e2e_step()
    s_out.wait_event(ev_done[(step_no[0] - 1) & 1])
    ev3.record(s_out)
    torch.cuda.synchronize(dev)
    barrier(pg)
    ms_e2e = max_over_ranks(pg, ev2.elapsed_time(ev3) / args.steps)
    h2d = sum(H[key].numel() * H[key].element_size() for key in inputs)
    d2h = H["o"].numel() * H["o"].element_size() + H["ht"].numel() * H["ht"].element_size()

    peak, peak_kind = load_peaks()
    abytes = algorithmic_bytes(x)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    kernel = "kda_recurrent_kernel" if args.entry == "recurrent" else forward_kernel(x, sms)
    launches = 1
    fused_here = kernel in ("kda_fwd_pc_kernel", "kda_fwd_tc_kernel", "kda_recurrent_kernel")
    if fe_on and (args.frontend == "unfused" or not fused_here):
        # the separate front-end pass: q and k norms, the gate, the beta sigmoid
        launches += 3 + (1 if x.beta is not None else 0)
        kernel = "front-end pass + " + kernel
    achieved = abytes / (ms / 1000.0) / 1e9
    traffic = None
    if args.frontend == "none" and kernel in KERNEL_SOURCES:
        traffic = MEASURED_TRAFFIC.get((args.workload, kernel_source_hash(kernel)))
    flops = algorithmic_flops(x)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import oracle_threads

        n_units = min(64, x.N * x.H_v)  # about 15-30 s of CPU work (0.25 s per unit-core of 8192 tokens)
        dt_cpu, tok_cpu, used = oracle_sample(x, n_units)
        cpu = {"value": tok_cpu / dt_cpu, "unit": "tokens/s", "cores": used, "kind": "oracle",
               "sample": f"{n_units} of {x.N * x.H_v} (sequence, head) units of {args.workload} "
                         f"({T} tokens each), fp64 token recurrence, {dt_cpu:.1f} s wall on "
                         f"{oracle_threads()} host threads"}

    if rank == 0:
        line = {
            "metric": metric_name(args.entry, args.workload), "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": x.dtype, "data": "synthetic",
            "config": {"workload": args.workload, "B": B, "T": T if not x.varlen else None,
                       "T_total": x.T_total, "H_k": x.H_k, "H_v": x.H_v, "d_k": x.d_k,
                       "d_v": x.d_v, "C": 64 if args.entry == "chunk" else None, "entry": args.entry,
                       "gate": "per-channel" if x.gate == "channel" else "per-head",
                       "beta": x.beta is not None, "h0": x.h0 is not None, "ht": True,
                       "frontend": args.frontend,
                       "global_batch": B * world, "seq_len": T if not x.varlen else x.T_total // B,
                       "parallelism": f"dp{world} (independent batches)",
                       "l2": f"inputs larger than L2 ({abytes / 1e6:.0f} MB per step), no flush"
                       if abytes > 129e6 else f"{abytes / 1e6:.0f} MB per step (not flushed)"},
            "e2e": {"value": tokens * world / (ms_e2e / 1000.0), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "schedule": "double-buffered: step i+1's H2D and step i-1's D2H overlap step i"},
            "ms_median_per_step": max_over_ranks(pg, ms_median),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic, "peak_kind": peak_kind,
                         "peak_nominal": NOMINAL_HBM_GBS, "frac_nominal": achieved / NOMINAL_HBM_GBS,
                         "frac_median": abytes / (ms_median / 1000.0) / 1e9 / peak,
                         "algorithmic_bytes_per_launch": abytes,
                         "kernel": kernel, "tflops": flops / (ms / 1000.0) / 1e12},
            "cpu_baseline": cpu,
            "clocks": clocks,
            "gpu_launches": args.steps * launches,
        }
        print(json.dumps(line), flush=True)


# The backward's contractions run on the tensor cores in tf32 (split operands, three
# products each). Their peak is the measured bf16 dense rate times the nominal tf32 / bf16
# ratio (1.1 / 2.25 PFLOP/s dense on GB300).
TF32_OVER_BF16 = 1.1 / 2.25


def tf32_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]) * TF32_OVER_BF16, "measured bf16 x nominal tf32/bf16 ratio"
    return 1900.0 * TF32_OVER_BF16, "fallback bf16 x nominal tf32/bf16 ratio"


def run_backward(args, world, rank, local, pg):
    """--entry backward: one kda_chunk_bwd call per step (the workload's forward inputs,
    a seeded dO and dht; all six gradients written)."""
    import numpy as np
    import torch

    from chunkwise_gated_linear_gb300 import kda
    from inputs import workload_inputs

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lib = kda.lib()
    x = workload_inputs(args.workload, seed=1000 + rank)
    B = x.N
    Bp = 1 if x.varlen else B
    T = x.T_total // Bp
    dt_io = torch.bfloat16 if x.dtype == "bf16" else torch.float32
    rng = np.random.default_rng(2000 + rank)

    def host(a, dtype, shape):
        return torch.from_numpy(np.ascontiguousarray(a)).reshape(shape).to(dtype).pin_memory()

    gshape = (Bp, T, x.H_v, x.d_k) if x.gate == "channel" else (Bp, T, x.H_v)
    H = {"q": host(x.q, dt_io, (Bp, T, x.H_k, x.d_k)), "k": host(x.k, dt_io, (Bp, T, x.H_k, x.d_k)),
         "v": host(x.v, dt_io, (Bp, T, x.H_v, x.d_v)), "g": host(x.g, torch.float32, gshape),
         "dO": host(rng.standard_normal(x.v.shape, dtype=np.float32), dt_io, (Bp, T, x.H_v, x.d_v)),
         "dht": host(rng.standard_normal((B, x.H_v, x.d_k, x.d_v), dtype=np.float32), torch.float32,
                     (B, x.H_v, x.d_k, x.d_v))}
    if x.beta is not None:
        H["beta"] = host(x.beta, torch.float32, (Bp, T, x.H_v))
    if x.h0 is not None:
        H["h0"] = host(x.h0, torch.float32, (B, x.H_v, x.d_k, x.d_v))
    inputs = [key for key in ("q", "k", "v", "g", "beta", "h0", "dO", "dht") if key in H]
    D = {key: t.to(dev) for key, t in H.items()}
    outs = {"dq": D["q"], "dk": D["k"], "dv": D["v"], "dg": D["g"], "dbeta": D.get("beta"), "dh0": D["dht"]}
    for key, like in outs.items():
        if like is not None:
            D[key] = torch.empty_like(like)
            H[key] = torch.empty_like(like, device="cpu").pin_memory()
    results = [key for key in outs if key in D]
    cu = torch.from_numpy(x.cu_seqlens.astype(np.int32)).to(dev) if x.varlen else None
    stream = torch.cuda.Stream(device=dev)
    sh = stream.cuda_stream
    ptr = lambda key: D[key].data_ptr() if key in D else None  # noqa: E731
    params = kda.kda_bwd_params(
        ptr("q"), ptr("k"), ptr("v"), ptr("g"), ptr("beta"), ptr("h0"), ptr("dO"), ptr("dht"), ptr("dq"), ptr("dk"),
        ptr("dv"), ptr("dg"), ptr("dbeta"), ptr("dh0"), B, T, x.H_k, x.H_v, x.d_k, x.d_v, 64, x.scale,
        None if cu is None else cu.data_ptr(), kda.KDA_DTYPE_BF16 if x.dtype == "bf16" else kda.KDA_DTYPE_F32,
        kda.KDA_GATE_PER_CHANNEL if x.gate == "channel" else kda.KDA_GATE_PER_HEAD, 0)

    def call():
        st = lib.kda_chunk_bwd(ctypes.byref(params), sh)
        if st != 0:
            raise RuntimeError(kda.status_string(st))

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev_step = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    with ClockSampler(local) as clk:
        barrier(pg)
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        for i in range(args.steps):
            ev_step[i].record(stream)
            call()
        ev_step[args.steps].record(stream)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(pg)
    ms = ev0.elapsed_time(ev1) / args.steps
    ms_median = statistics.median(ev_step[i].elapsed_time(ev_step[i + 1]) for i in range(args.steps))
    clocks = clk.summary()
    ms_max = max_over_ranks(pg, ms)

    def e2e_step():
        with torch.cuda.stream(stream):
            for key in inputs:
                D[key].copy_(H[key], non_blocking=True)
            call()
            for key in results:
                H[key].copy_(D[key], non_blocking=True)

    for _ in range(max(1, args.warmup // 2)):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(pg)
    ev2, ev3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev2.record(stream)
    for _ in range(args.steps):
        e2e_step()
    ev3.record(stream)
    torch.cuda.synchronize(dev)
    barrier(pg)
    ms_e2e = max_over_ranks(pg, ev2.elapsed_time(ev3) / args.steps)
    h2d = sum(H[key].numel() * H[key].element_size() for key in inputs)
    d2h = sum(H[key].numel() * H[key].element_size() for key in results)

    flops = backward_flops(x)
    tflops = flops / (ms / 1000.0) / 1e12
    peak, tc_kind = tf32_peak()
    hbm_peak, peak_kind = load_peaks()
    abytes = backward_bytes(x)
    if rank == 0:
        tokens = x.T_total
        line = {
            "metric": metric_name("backward", args.workload), "value": tokens * world / (ms_max / 1000.0),
            "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": args.workload, "entry": "backward", "B": B, "T_total": x.T_total,
                       "H_k": x.H_k, "H_v": x.H_v, "d_k": x.d_k, "d_v": x.d_v, "C": 64,
                       "io_dtype": x.dtype, "gate": "per-channel" if x.gate == "channel" else "per-head",
                       "beta": x.beta is not None, "h0": x.h0 is not None, "dht": True,
                       "global_batch": B * world, "parallelism": f"dp{world} (independent batches)",
                       "l2": f"inputs larger than L2 ({abytes / 1e6:.0f} MB per step), no flush"},
            "e2e": {"value": tokens * world / (ms_e2e / 1000.0), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "ms_median_per_step": max_over_ranks(pg, ms_median),
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                         "frac": tflops / peak, "traffic": None, "peak_kind": tc_kind,
                         "algorithmic_flops_per_launch": flops, "kernel": "backward (prep, states, adjoint, grads, finish)",
                         "hbm_bytes_per_launch": abytes, "hbm_frac": abytes / (ms / 1000.0) / 1e9 / hbm_peak},
            "cpu_baseline": None,
            "clocks": clocks,
            "gpu_launches": args.steps * (6 if (x.dtype == "bf16" and x.H_v != x.H_k) else 4),
        }
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--entry", choices=["chunk", "recurrent", "backward"], default="chunk",
                    help="kda_chunk_fwd (default), kda_recurrent_fwd (the token-by-token decode step) "
                         "or kda_chunk_bwd (the backward pass)")
    ap.add_argument("--frontend", choices=["none", "fused", "unfused"], default="none",
                    help="raw q, k, gate pre-activations and beta logits through the front-end "
                         "(q/k L2 norm, gated gate, beta sigmoid): applied inside the forward kernel "
                         "where it can (fused) or as a separate pass (unfused)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # the timing rules ask for at least 3 warm-up steps
    world, rank, local, pg = dist_setup()
    try:
        if args.impl == "reference":
            run_reference(args, world, rank, pg)
        else:
            (run_backward if args.entry == "backward" else run_ours)(args, world, rank, local, pg)
    finally:
        if pg is not None:
            pg.destroy_process_group()


if __name__ == "__main__":
    main()
