#!/usr/bin/env python3
"""Throughput of chunked KDA prefill on GB300, one JSON line on stdout.

A step is one kda_chunk_prefill call (prologue when packed, intra-chunk
kernel, recurrent kernel) over one batch of the workload, inputs resident in
HBM. ``--impl reference`` times the fp64 CPU oracle instead, on a bounded
sample of the same workload. Under torchrun every rank runs its own copy of
the workload on its own GPU (weak scaling, no collective on the data path).
"""
import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import kda_inputs as KI  # noqa: E402

METRIC = "KDA prefill tokens/s (T=8192, H=64, D=128) on 1 GB300; % of roofline"
UNIT = "tokens/s"

# Counted work of the chunked algorithm (dense 16-token tiles, 2 FLOP/MAC).
FLOPS_INTRA_PER_CHUNK_HEAD = 262144 + 2731     # gated Gram + scores, W, Ut; inversion
FLOPS_RECUR_PER_CHUNK_HEAD = 1638400           # W S, Qg S, P U, Kd^T U
# 64-token path, per (64-token chunk, head): the chain's W S, Qg S, P U and
# Kd^T U (2 x 64 x 128 x 128 each, P U 2 x 64 x 64 x 128); the record
# builder's Gram and scores (2 x 128 x 64 x 128), W and Ut (2 x 64 x 64 x 128
# each) and the 64 x 64 inversion (64^3 / 3)
FLOPS_C64_CHAIN_PER_CHUNK_HEAD = 3 * 2097152 + 1048576
FLOPS_C64_INTRA_PER_CHUNK_HEAD = 2097152 + 2 * 1048576 + 87381
FLOPS_C64_PER_CHUNK_HEAD = FLOPS_C64_CHAIN_PER_CHUNK_HEAD + FLOPS_C64_INTRA_PER_CHUNK_HEAD
BYTES_IN_PER_TOKEN_HEAD = 3 * 256 + 512 + 4    # q, k, v bf16; g fp32; beta fp32
BYTES_OUT_PER_TOKEN_HEAD = 256                 # o bf16
STATE_BYTES = 128 * 128 * 4


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 2000 for the CUDA path, about 1 s on the headline "
                         "workload; 50 for the reference arm)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=KI.HEADLINE, choices=KI.WORKLOAD_ORDER)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--recurrent-impl", type=int, default=None,
                    help="1 = 16-token chunks, 3 = 64-token chunks on tcgen05 (two kernels), "
                         "4 = 64-token chunks in one cooperative launch (library default if unset)")
    ap.add_argument("--decode", default=None, metavar="NxH",
                    help="time the one-token decode step instead (e.g. 256x64) and print its line")
    ap.add_argument("--preprocess", action="store_true",
                    help="run the prefill with the in-kernel input preprocessing on (q/k "
                         "normalisation, g read as gate logits): the same inputs, for timing")
    ap.add_argument("--no-decode", action="store_true",
                    help="leave the decode measurement out of the default line")
    ap.add_argument("--backward-impl", type=int, default=0, choices=[0, 1],
                    help="gradient form for --backward: 0 chunked (default), 1 token-serial")
    ap.add_argument("--backward", action="store_true",
                    help="time the gradient call (kda_chunk_prefill_backward) on the workload "
                         "instead of the prefill; prints its own line")
    ap.add_argument("--gate-mu", type=float, default=None,
                    help="mean of the gate pre-activation (g = logsigmoid(N(mu, 1))) instead of "
                         "the workload's; about -6 or below puts every chunk-head outside the "
                         "factored range (the exact form)")
    ap.add_argument("--scan-segments", type=int, default=None,
                    help="segments of the 16-token path's segment-parallel scan (0 = automatic, "
                         "1 = off; library default if unset)")
    ap.add_argument("--heads", type=int, default=None,
                    help="run the workload with this many heads instead (a smaller case for "
                         "profiler captures; the line's config then says so)")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = 2000 if args.impl == "ours" else 50
    return args


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def workload_counts(d, H):
    lens = d["seqlens"]
    tokens = sum(lens)
    chunks = sum((L + 15) // 16 for L in lens)
    n = len(lens)
    init = d["initial_state"] is not None
    intra_bytes = tokens * H * BYTES_IN_PER_TOKEN_HEAD
    recur_bytes = tokens * H * BYTES_OUT_PER_TOKEN_HEAD + n * H * STATE_BYTES * (1 + int(init))
    c64 = sum((L + 63) // 64 for L in lens)
    return dict(tokens=tokens, chunk_heads=chunks * H, n_seqs=n, c64_chunk_heads=c64 * H,
                intra_bytes=intra_bytes, recur_bytes=recur_bytes,
                path_bytes=intra_bytes + recur_bytes,
                intra_flops=chunks * H * FLOPS_INTRA_PER_CHUNK_HEAD,
                recur_flops=chunks * H * FLOPS_RECUR_PER_CHUNK_HEAD)


class ClockSampler:
    """nvidia-smi samples every 100 ms while the timed loops run."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.samples, self.proc, self.thread = [], None, None
        self.sel = []
        try:
            bus = torch.cuda.get_device_properties(device).pci_bus_id
            dom = torch.cuda.get_device_properties(device).pci_domain_id
            dv = torch.cuda.get_device_properties(device).pci_device_id
            self.sel = ["-i", f"{dom:08X}:{bus:02X}:{dv:02X}.0"]
        except Exception:
            self.sel = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", *self.sel, f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == 7:
                self.samples.append(parts)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, reasons = [], None, set()
        for s in self.samples:
            try:
                sm.append(float(s[0]))
                mx = float(s[1])
            except ValueError:
                continue
            for nm, val in zip(names, s[3:]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def scan_segments(n_units, chunks, sms):
    """Segments of the 16-token path's segment-parallel scan for fixed-length
    calls, as the library picks them (automatic setting)."""
    if chunks < 64 or 4 * n_units > sms - 4:
        return 1
    P = min(3 * (sms - 4) // (2 * n_units), 16, chunks // 16)
    if P < 2:
        return 1
    L = -(-chunks // P)
    return -(-chunks // L)


def launches_per_call(w, args):
    """Kernels one prefill call launches. 16-token path: the cu_seqlens
    prologue (packed batches), the intra-chunk kernel, its exact-form
    companion, the recurrent kernel, and for long fixed-length sequences with
    few heads the segment scan's maps launch and (P > 2) its combine.
    64-token paths: the prologue (packed), then the intra-chunk and recurrent
    kernels (split) or the one cooperative kernel (fused)."""
    impl = 1 if args.recurrent_impl is None else args.recurrent_impl
    if impl == 3:
        return 2 + int(w.varlen)
    if impl == 4:
        return 1 + int(w.varlen)
    n = 3 + int(w.varlen)
    chunks = -(-(w.T // w.n_seqs) // 16)
    sms = (torch.cuda.get_device_properties(0).multi_processor_count
           if torch.cuda.is_available() else 152)
    if not w.varlen:
        P = scan_segments(w.n_seqs * w.H, chunks, sms)
        n += (P >= 2) + (P > 2)
    return n


def stock_workload(args):
    """Whether the run is the named workload with no size, gate, input
    preprocessing or scan override (the traffic records are per workload as
    named)."""
    return (args.heads is None and args.gate_mu is None and not args.preprocess
            and args.scan_segments is None)


def traffic_for(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on this kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(kernel)
    if not rec:
        return None
    srcs = rec["source"] if isinstance(rec["source"], list) else [rec["source"]]
    h = hashlib.sha256()
    for f in srcs:   # the kernel's file and the headers holding its body
        h.update(open(os.path.join(ROOT, "prefill_kda_chunk_gb300", "csrc", f), "rb").read())
    sha = h.hexdigest()[:16]
    if sha != rec.get("source_sha") or workload not in rec.get("per_launch_bytes", {}):
        return None
    return rec["per_launch_bytes"][workload]


def run_reference(args, rank, world):
    """fp64 CPU oracle, bounded sample of the workload per step, rank 0 only."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = KI.WORKLOADS[args.workload]
    if args.gate_mu is not None:
        w = dataclasses.replace(w, mu=args.gate_mu)
    if args.heads is not None:
        w = dataclasses.replace(w, H=args.heads)
    d = KI.make_inputs(w)
    cores = len(os.sched_getaffinity(0))
    # one head per host core (the oracle runs one (sequence, head) per thread);
    # a single long sequence is cut to a prefix so that a step stays near half
    # a second (~63 us per token-head per core for the fp64 recurrence)
    Hs = max(1, min(w.H, cores))
    Ts = w.T
    if len(d["seqlens"]) == 1:
        Ts = max(16, min(w.T, int(0.5 * cores / 63e-6 / Hs)))
    sub = {n: d[n][:Ts, :Hs].contiguous() for n in ("q", "k", "v", "g", "beta")}
    s0 = None if d["initial_state"] is None else d["initial_state"][:, :Hs].contiguous()
    cu = d["cu_seqlens"] if Ts == w.T else torch.tensor([0, Ts], dtype=torch.int32)

    def step():
        oracle.recurrent(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], initial_state=s0,
                         cu_seqlens=cu, scale=d["scale"], out_tokens=Ts, threads=cores)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    tokens_equiv = Ts * Hs / w.H           # one step covers Hs of the H heads, Ts tokens
    value = args.steps * tokens_equiv / dt
    sample = (f"{Hs} of {w.H} heads, " +
              (f"all {w.T} tokens" if Ts == w.T else f"the first {Ts} of {w.T} tokens") +
              f", per step, {Hs} threads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(w, d),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_of(w, d):
    return {"workload": w.name, "T": w.T, "H": w.H, "D": 128, "n_seqs": len(d["seqlens"]),
            "initial_state": d["initial_state"] is not None, "seed": w.seed,
            "gate_mu": w.mu, "l2": "inputs larger than L2, no flush between steps"}


def cpu_baseline(w, d):
    import oracle
    oracle.build()
    cores = len(os.sched_getaffinity(0))
    # about 30 core-seconds: ~63 us per token-head per core for the fp64 recurrence
    Hs = max(1, min(w.H, int(30.0 / (w.T * 63e-6))))
    sub = {n: d[n][:, :Hs].contiguous() for n in ("q", "k", "v", "g", "beta")}
    s0 = None if d["initial_state"] is None else d["initial_state"][:, :Hs].contiguous()
    t0 = time.perf_counter()
    oracle.recurrent(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], initial_state=s0,
                     cu_seqlens=d["cu_seqlens"], scale=d["scale"], threads=cores)
    dt = time.perf_counter() - t0
    return {"value": w.T * Hs / w.H / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{Hs} of {w.H} heads x {w.T} tokens, {dt:.2f} s wall"}


DECODE_BYTES = 4 * 256 + 512 + 4 + 2 * 128 * 128 * 4   # per (sequence, head): q k v o, g, beta, S in+out


def bench_decode(K, dev, N, H, steps, warmup, hbm):
    """Decode steps in place on a resident batch (state > L2), CUDA events."""
    d = KI.make_case([1] * N, H=H, seed=9, init_state=True)
    x = {n: d[n].to(dev) for n in ("q", "k", "v", "g", "beta")}
    state = d["initial_state"].to(dev)
    out = torch.empty_like(x["v"])
    stream = torch.cuda.current_stream(dev)

    def step():
        K.decode_step(x["q"], x["k"], x["v"], x["g"], x["beta"], state=state, scale=d["scale"],
                      out=out, in_place=True)

    for _ in range(max(warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(b) / steps
    gbs = N * H * DECODE_BYTES / (ms / 1e3) / 1e9
    return {"workload": f"decode_N{N}_H{H}", "tokens_per_s": N / (ms / 1e3),
            "token_heads_per_s": N * H / (ms / 1e3), "us_per_step": 1e3 * ms, "steps": steps,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                         "frac": gbs / hbm, "bytes_per_step": N * H * DECODE_BYTES}}


# algorithmic bytes of the gradient call: per token-head q, k, v, dO (bf16)
# and g, beta read, dq, dk, dv, dg, dbeta written (fp32); per (sequence, head)
# the initial state and dL/d(final state) read and dL/d(initial state) written
BWD_TOKEN_HEAD_BYTES = 4 * 128 * 2 + 128 * 4 + 4 + 4 * 128 * 4 + 4
BWD_UNIT_BYTES = 3 * 128 * 128 * 4


def bench_backward(K, dev, w, args, hbm):
    """The gradient call on the workload's inputs (resident), CUDA events;
    plus the fp64 gradient oracle on a bounded sample of host work."""
    d = KI.make_inputs(w)
    H, T = w.H, w.T
    gen = torch.Generator().manual_seed(w.seed + 7)
    n_seqs = len(d["seqlens"])
    dout = torch.randn(T, H, 128, generator=gen).to(torch.bfloat16)
    dsf = torch.randn(n_seqs, H, 128, 128, generator=gen) * 0.1
    x = {n: d[n].to(dev) for n in ("q", "k", "v", "g", "beta")}
    s0 = None if d["initial_state"] is None else d["initial_state"].to(dev)
    cu = d["cu_seqlens"].to(dev) if w.varlen else None
    if not w.varlen:
        x = {n: t.view(1, T, *t.shape[1:]) for n, t in x.items()}
    do_d, dsf_d = dout.to(dev).view(x["v"].shape), dsf.to(dev)
    stream = torch.cuda.current_stream(dev)

    K.kda_set_backward_impl(args.backward_impl)

    def call():
        return K.chunk_prefill_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], do_d,
                                        initial_state=s0, cu_seqlens=cu, scale=d["scale"],
                                        d_final_state=dsf_d)

    clocks = ClockSampler(dev)
    clocks.start()
    for _ in range(max(args.warmup, 3)):
        call()
    K.check_device_error()
    torch.cuda.synchronize(dev)
    steps = args.steps
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        call()
    b.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    K.check_device_error()
    ms = a.elapsed_time(b) / steps
    nbytes = T * H * BWD_TOKEN_HEAD_BYTES + n_seqs * H * BWD_UNIT_BYTES
    gbs = nbytes / (ms / 1e3) / 1e9
    line = {"metric": f"KDA prefill backward tokens/s (T={T}, H={H}, D=128) on 1 GB300",
            "value": T / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "dtype": "fp32 (bf16 q, k, v, dO)", "data": "synthetic",
            "config": dict(config_of(w, d), backward=True),
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                         "frac": gbs / hbm,
                         # DRAM bytes of the whole chunked call (all its launches), from
                         # the committed ncu record
                         "traffic": (traffic_for("backward_call", w.name)
                                     if args.backward_impl == 0 and stock_workload(args) else None),
                         "kernel": ("the whole call: intra-chunk, exact form, both chains, gradients"
                                    if args.backward_impl == 0 else "kda_backward_kernel"),
                         "bytes_per_call": nbytes},
            "backward_impl": "chunked" if args.backward_impl == 0 else "token-serial",
            "clocks": clk,
            # chunked: intra-chunk, exact form, the chains, the gradient kernel
            "gpu_launches": steps * ((4 if args.backward_impl == 0 else 1) + int(w.varlen))}
    if not args.no_cpu_baseline:
        import oracle
        oracle.build()
        cores = len(os.sched_getaffinity(0))
        # one (sequence, head) per host thread; ~0.2 ms of fp64 work per token-head
        Hs, Ts = min(H, cores), min(d["seqlens"][0], 1024)
        sub = {n: d[n][:Ts, :Hs] for n in ("q", "k", "v", "g", "beta")}
        t0 = time.perf_counter()
        oracle.recurrent_backward(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"],
                                  dout[:Ts, :Hs], scale=d["scale"], threads=cores)
        sec = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": Ts * Hs / H / sec, "unit": "tokens/s",
                                "cores": min(cores, Hs), "kind": "oracle",
                                "sample": f"{Hs} of {H} heads x {Ts} tokens, {sec:.2f} s wall"}
    return line


def main():
    args = parse()
    rank, world, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    import prefill_kda_chunk_gb300 as K
    from prefill_kda_chunk_gb300 import build as B
    if rank == 0:
        B.build()
    barrier(world)
    K.lib()
    if args.recurrent_impl is not None:
        K.kda_set_recurrent_impl(args.recurrent_impl)
    if args.scan_segments is not None:
        K.kda_set_scan_segments(args.scan_segments)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if args.decode:
        Nd, Hd = (int(v) for v in args.decode.lower().split("x"))
        hbm, _, _ = load_peaks()
        r = bench_decode(K, dev, Nd, Hd, min(args.steps, 500), args.warmup, hbm)
        if rank == 0:
            print(json.dumps({"metric": f"KDA decode tokens/s (one token per sequence, N={Nd}, "
                                        f"H={Hd}, D=128) on 1 GB300",
                              "value": world * r["tokens_per_s"], "unit": "tokens/s",
                              "n_gpus": world, "higher_is_better": True, "dtype": "bf16",
                              "data": "synthetic", **r}), flush=True)
        return

    w = KI.WORKLOADS[args.workload]
    if args.gate_mu is not None:
        w = dataclasses.replace(w, mu=args.gate_mu)
    if args.heads is not None:
        w = dataclasses.replace(w, H=args.heads)
    if args.backward:
        hbm, _, _ = load_peaks()
        line = bench_backward(K, dev, w, args, hbm)
        if rank == 0:
            print(json.dumps(line), flush=True)
        return
    d = KI.make_inputs(w)
    H = w.H
    cnt = workload_counts(d, H)
    x = {n: d[n].to(dev) for n in ("q", "k", "v", "g", "beta")}
    s0 = None if d["initial_state"] is None else d["initial_state"].to(dev)
    cu = d["cu_seqlens"].to(dev) if w.varlen else None
    out = torch.empty_like(x["v"])
    fin = torch.empty((cnt["n_seqs"], H, 128, 128), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call(q=x["q"], k=x["k"], v=x["v"], g=x["g"], beta=x["beta"], s0=s0, cu=cu, out=out):
        K.chunk_prefill(q, k, v, g, beta, initial_state=s0, cu_seqlens=cu, scale=d["scale"],
                        out=out, final_state=fin, normalize_qk=args.preprocess,
                        gate_logits=args.preprocess)

    clocks = ClockSampler(dev)
    clocks.start()
    for _ in range(max(args.warmup, 3)):
        call()
    K.check_device_error()
    torch.cuda.synchronize(dev)
    barrier(world)

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    barrier(world)
    start.record(stream)
    for i in range(args.steps):
        call()
    end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    K.check_device_error()
    ms = max_over_ranks(start.elapsed_time(end), world)
    clk = clocks.stop()
    # the split between the kernels, from events the library records around
    # them, in a second run of the same steps (the events sit between the
    # kernels, so they stay out of the headline timing above)
    if K.kda_stage_timing_begin(args.steps) != 0:
        raise RuntimeError("kda_stage_timing_begin failed")
    for i in range(args.steps):
        call()
    torch.cuda.synchronize(dev)
    rc, intra_ms, recur_ms, ncalls = K.kda_stage_timing_end()
    if rc != 0 or ncalls != args.steps:
        raise RuntimeError(f"stage timing failed ({rc}, {ncalls} calls)")

    # end to end: every step copies its inputs in from pinned host memory and its
    # results (o and the final state) back out. Steps are pipelined the way a
    # serving loop would run them: two device buffer sets, inputs of step i+1
    # copied in on two copy streams while step i computes and is read back.
    e2e = None
    if not args.no_e2e:
        names = ("q", "k", "v", "g", "beta")
        hin = {n: d[n].pin_memory() for n in names}
        hs0 = None if s0 is None else d["initial_state"].pin_memory()
        hcu = d["cu_seqlens"].pin_memory() if w.varlen else None
        nb = 2
        dset = [{n: torch.empty_like(x[n]) for n in names} for _ in range(nb)]
        ds0 = [None if s0 is None else torch.empty_like(s0) for _ in range(nb)]
        dcu = [None if cu is None else torch.empty_like(cu) for _ in range(nb)]
        dout = [torch.empty_like(out) for _ in range(nb)]
        dfin = [torch.empty_like(fin) for _ in range(nb)]
        hout = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(nb)]
        hfin = [torch.empty(fin.shape, dtype=fin.dtype).pin_memory() for _ in range(nb)]
        h2d = sum(t.numel() * t.element_size() for t in hin.values())
        h2d += 0 if hs0 is None else hs0.numel() * 4
        h2d += 0 if hcu is None else hcu.numel() * 4
        d2h = out.numel() * 2 + fin.numel() * 4
        # the two copy-in streams take about half of the input bytes each
        groups = (("g", "beta"), ("q", "k", "v"))
        s_in = [torch.cuda.Stream(dev) for _ in groups]
        s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = lambda: torch.cuda.Event()
        in_done = [[ev() for _ in range(nb)] for _ in groups]
        cmp_done = [ev() for _ in range(nb)]
        out_done = [ev() for _ in range(nb)]
        used = [False] * nb

        def e2e_step(i):
            b = i % nb
            for j, grp in enumerate(groups):
                st = s_in[j]
                if used[b]:
                    st.wait_event(cmp_done[b])        # buffer set b is no longer read
                with torch.cuda.stream(st):
                    for n in grp:
                        dset[b][n].copy_(hin[n], non_blocking=True)
                    if j == 0 and ds0[b] is not None:
                        ds0[b].copy_(hs0, non_blocking=True)
                    if j == 0 and dcu[b] is not None:
                        dcu[b].copy_(hcu, non_blocking=True)
                in_done[j][b].record(st)
            for j in range(len(groups)):
                s_cmp.wait_event(in_done[j][b])
            if used[b]:
                s_cmp.wait_event(out_done[b])         # o / state of step i-2 are read back
            with torch.cuda.stream(s_cmp):
                K.chunk_prefill(dset[b]["q"], dset[b]["k"], dset[b]["v"], dset[b]["g"],
                                dset[b]["beta"], initial_state=ds0[b], cu_seqlens=dcu[b],
                                scale=d["scale"], out=dout[b], final_state=dfin[b],
                                normalize_qk=args.preprocess, gate_logits=args.preprocess)
            cmp_done[b].record(s_cmp)
            s_out.wait_event(cmp_done[b])
            with torch.cuda.stream(s_out):
                hout[b].copy_(dout[b], non_blocking=True)
                hfin[b].copy_(dfin[b], non_blocking=True)
            out_done[b].record(s_out)
            used[b] = True

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        barrier(world)
        es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2e_steps = max(3, min(args.steps, 20))
        es.record(stream)
        for st in (*s_in, s_cmp, s_out):
            st.wait_event(es)
        for i in range(e2e_steps):
            e2e_step(i)
        for st in (*s_in, s_cmp, s_out):
            stream.wait_stream(st)
        ee.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        K.check_device_error()
        # the last step's results must match the resident run's
        if not (torch.equal(hout[(e2e_steps - 1) % nb], out.cpu())
                and torch.equal(hfin[(e2e_steps - 1) % nb], fin.cpu())):
            raise RuntimeError("end-to-end run differs from the resident run")
        ems = max_over_ranks(es.elapsed_time(ee), world)
        e2e = {"value": world * cnt["tokens"] * e2e_steps / (ems / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "pipelined": "2 buffer sets; copies of step i+1 overlap step i"}

    if rank != 0:
        return
    hbm, tf, peak_src = load_peaks()
    sec = ms / 1e3 / args.steps
    value = world * cnt["tokens"] * args.steps / (ms / 1e3)

    impl = 1 if args.recurrent_impl is None else args.recurrent_impl

    def hbm_kernel(ms_, nbytes, flops):
        gbs = nbytes / (ms_ / 1e3) / 1e9
        return {"ms": ms_, "bound": "hbm", "alg_bytes": nbytes, "alg_flops": flops,
                "achieved_gbs": gbs, "frac": gbs / hbm}

    def tc_kernel(ms_, nbytes, flops):
        tfs = flops / (ms_ / 1e3) / 1e12
        return {"ms": ms_, "bound": "tensor", "alg_bytes": nbytes, "alg_flops": flops,
                "achieved_tflops": tfs, "frac": tfs / tf}

    c64_chunk_heads = cnt["c64_chunk_heads"]
    if impl == 4:
        # one cooperative kernel: the whole path's bytes
        kernels = {"kda_c64_fused_kernel": hbm_kernel(recur_ms, cnt["path_bytes"],
                                                      c64_chunk_heads * FLOPS_C64_PER_CHUNK_HEAD)}
    elif impl == 3:
        kernels = {
            "kda_c64_intra_kernel": hbm_kernel(intra_ms, cnt["intra_bytes"],
                                               c64_chunk_heads * FLOPS_C64_INTRA_PER_CHUNK_HEAD),
            "kda_c64_chain_kernel": tc_kernel(recur_ms, cnt["recur_bytes"],
                                              c64_chunk_heads * FLOPS_C64_CHAIN_PER_CHUNK_HEAD)}
    else:
        kernels = {
            "kda_intra_chunk_kernel": hbm_kernel(intra_ms, cnt["intra_bytes"], cnt["intra_flops"]),
            "kda_recurrent_kernel": tc_kernel(recur_ms, cnt["recur_bytes"], cnt["recur_flops"])}
    dom = max(kernels, key=lambda k: kernels[k]["ms"])
    kd = kernels[dom]
    if kd["bound"] == "hbm":
        roof = {"bound": "hbm", "achieved": kd["achieved_gbs"], "peak": hbm, "unit": "GB/s",
                "frac": kd["frac"]}
    else:
        roof = {"bound": "tensor", "achieved": kd["achieved_tflops"], "peak": tf,
                "unit": "TFLOP/s", "frac": kd["frac"]}
    roof.update({"kernel": dom, "peak_source": f"{peak_src} (MEASURED_PEAKS.json burst)"
                 if peak_src == "measured" else "fallback",
                 # a record holds for the workload it was captured on, as it is
                 "traffic": traffic_for(dom, w.name) if stock_workload(args) else None})
    # the whole call against the slower of the two bounds of the counted work
    t_hbm = cnt["path_bytes"] / (hbm * 1e9)
    t_tc = (cnt["intra_flops"] + cnt["recur_flops"]) / (tf * 1e12)
    path_roof = {"bound": "hbm" if t_hbm >= t_tc else "tensor", "roofline_us": 1e6 * max(t_hbm, t_tc),
                 "measured_us": 1e6 * sec, "frac": max(t_hbm, t_tc) / sec,
                 "alg_bytes": cnt["path_bytes"],
                 "alg_flops": cnt["intra_flops"] + cnt["recur_flops"],
                 "achieved_gbs": cnt["path_bytes"] / sec / 1e9}

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict(config_of(w, d), **({"preprocess": "q/k norm + gate logits in-kernel"}
                                                if args.preprocess else {})),
            "roofline": roof, "path_roofline": path_roof,
            "kernels": kernels, "gpu_launches": args.steps * launches_per_call(w, args),
            "clocks": clk, "e2e": e2e}
    if not args.no_decode:
        line["decode"] = bench_decode(K, dev, 256, 64, 200, args.warmup, hbm)
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(w, d)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
