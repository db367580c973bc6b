#!/usr/bin/env python
"""Benchmark of the chunked gated delta rule operator on one GB300.

One step = the whole hot path over one batch, as a training step runs it:
gdn_chunk_fwd_save (output, final state, and every chunk's start state and T
tiles kept for the backward) followed by gdn_chunk_bwd_saved (upstream
dO ~ N(0,1)) on the dense workload B=4, H=16, T=4096, d_k=d_v=128 (bf16 I/O,
fp32 state), inputs resident in HBM.  The inference forward (gdn_chunk_fwd,
nothing kept) is timed beside it.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle on the host cores (bounded
samples of the same workload); it is the only other place besides the
cpu_baseline leg where this script runs the oracle.

Multi-GPU (torchrun, one rank per GPU): every rank runs its own batch of the
same shape (independent problems, no data-path collective; weak scaling);
the barrier and the max-over-ranks reduction of the step time are the only
communication.
"""

from __future__ import annotations

import argparse
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

METRIC = "GDN chunk fwd/bwd tokens·heads/s on 1 GB300; % of roofline; rel-RMS vs oracle"
UNIT = "tokens·heads/s"
SHAPE = dict(B=4, T=4096, H=16, d_k=128, d_v=128)
CHUNK = 64
L2_BYTES = 129 * 2**20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------
# algorithmic work per token-head (C = 64): fixed formulas, frozen before tuning
# ----------------------------------------------------------------------------

def fwd_flops(K, V, C=CHUNK):
    return 6 * K * V + 3 * C * K + 2 * C * V + C * C / 3.0


def fwd_bytes(K, V):
    return 4 * K + 4 * V + 6


def bwd_flops(K, V, C=CHUNK):
    return 16 * K * V + 9 * C * K + 6 * C * V + C * C


def bwd_bytes(K, V):
    return 8 * K + 6 * V + 12


def workload_totals(B, T, H, K, V):
    th = B * T * H
    units = B * H
    f_fwd = fwd_flops(K, V) * th
    b_fwd = fwd_bytes(K, V) * th + 4 * K * V * units          # + final state write
    f_bwd = bwd_flops(K, V) * th
    b_bwd = bwd_bytes(K, V) * th
    return th, f_fwd, b_fwd, f_bwd, b_bwd


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------
# distributed plumbing
# ----------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def rank_seed(rank):
    """Seed of rank r's batch: every rank draws its own independent problems."""
    return 2 + 1000 * rank


def aggregate_rate(world, units_per_rank, t_max):
    """Whole-job throughput: the units all ranks processed over the slowest
    rank's time (weak scaling, each rank holds a batch of the same shape)."""
    return world * units_per_rank / t_max


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.2)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append(dict(sm=float(parts[1]), sm_max=float(parts[2]),
                                     power=float(parts[3]), hw=parts[5], hw_thermal=parts[6],
                                     sw_thermal=parts[7], sw_power=parts[8]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        busy = [r for r in rows if r["power"] > 0.25 * max(x["power"] for x in rows)] or rows
        return {"sm_mhz": statistics.median(r["sm"] for r in busy),
                "sm_max_mhz": max(r["sm_max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


# ----------------------------------------------------------------------------
# CPU oracle legs
# ----------------------------------------------------------------------------

def oracle_sample(wl, budget_s, threads):
    """Time the fp64 oracle (forward + reverse mode) on (batch, head) units of
    ``wl`` in waves of ``threads`` units until ``budget_s`` is spent.
    Returns (token_heads, seconds, units, results)."""
    from oracle import recurrence
    units_all = [(s, h) for s in range(wl.n_seq) for h in range(wl.H)]
    done = []
    t0 = time.perf_counter()
    fwd_res = None
    bwd_res = None
    i = 0
    while i < len(units_all):
        wave = units_all[i:i + threads]
        o, S = recurrence.workload_fwd(wl, units=wave, threads=threads)
        g = recurrence.workload_bwd(wl, units=wave, threads=threads)
        if fwd_res is None:
            fwd_res, bwd_res = (o, S), g
        else:
            for (s, h) in wave:
                fwd_res[0][s, :, h] = o[s, :, h]
                fwd_res[1][s, h] = S[s, h]
                for n in g:
                    if n == "dS0":
                        bwd_res[n][s, h] = g[n][s, h]
                    else:
                        bwd_res[n][s, :, h] = g[n][s, :, h]
        done += wave
        i += threads
        if time.perf_counter() - t0 >= budget_s:
            break
    secs = time.perf_counter() - t0
    th = sum(wl.T for _ in done)
    return th, secs, done, fwd_res, bwd_res


def run_reference(args):
    """--impl reference: the oracle as it stands, on the host cores."""
    world, rank, _ = dist_env()
    if world > 1 and rank != 0:
        return 0
    from linear_attention_sequence_chunked_gb300 import workloads as W
    from oracle import recurrence
    recurrence.build_oracle()
    threads = recurrence.default_threads()
    wl = W.make_workload(2, with_grad=True, **{k: SHAPE[k] for k in ("B", "T", "H", "d_k", "d_v")})
    units_all = [(s, h) for s in range(wl.n_seq) for h in range(wl.H)]
    per_step = min(len(units_all), threads)
    times = []
    for i in range(args.warmup + args.steps):
        j = (i * per_step) % len(units_all)
        wave = (units_all + units_all)[j:j + per_step]
        t0 = time.perf_counter()
        recurrence.workload_fwd(wl, units=wave, threads=threads)
        recurrence.workload_bwd(wl, units=wave, threads=threads)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    step_s = statistics.mean(times)
    th = per_step * wl.T
    value = th / step_s
    sample = (f"{per_step} (batch, head) units of T={wl.T} per step (fwd + reverse mode), "
              f"fp64, {threads} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "dense fwd+bwd B=4 H=16 T=4096 d_k=128 d_v=128 (sampled units)",
                   "global_batch": SHAPE["B"], "seq_len": SHAPE["T"], "heads": SHAPE["H"],
                   "d_k": SHAPE["d_k"], "d_v": SHAPE["d_v"], "parallelism": "host threads"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------
# GPU leg
# ----------------------------------------------------------------------------

def _bf16(a, torch, dev):
    import numpy as np
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)


def run_ours(args):
    import numpy as np
    import torch

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")

    from linear_attention_sequence_chunked_gb300 import build as libbuild
    from linear_attention_sequence_chunked_gb300 import gdn
    from linear_attention_sequence_chunked_gb300 import workloads as W
    if rank == 0:
        libbuild.build()
    barrier(world)
    libbuild.build()
    gdn.load()

    if args.split_only:
        # profiling aid: only the sequence-split measurement at one segment
        # count (one warm-up and one timed call per route), printed as JSON
        if rank == 0:
            r = measure_split(gdn, torch, dev, torch.cuda.current_stream(), segs=(args.split_only,), steps=1,
                              warmup=1)
            print(json.dumps(r))
        return 0

    if args.kda_once:
        # profiling aid: one per-channel-gate forward (workspace route) and
        # one backward at B,H,T (d_k = d_v = 128), printed as JSON
        if rank == 0:
            kb, kh, kt = (int(x) for x in args.kda_once.split(","))
            print(json.dumps(measure_kda(gdn, torch, dev, torch.cuda.current_stream(), None, B=kb, H=kh, T=kt,
                                         once=True)))
        return 0

    B, T, H, K, V = (SHAPE[k] for k in ("B", "T", "H", "d_k", "d_v"))
    wl = W.make_workload(2, B=B, T=T, H=H, d_k=K, d_v=V, with_grad=True,
                         seed=rank_seed(rank))
    q, k, v = _bf16(wl.q, torch, dev), _bf16(wl.k, torch, dev), _bf16(wl.v, torch, dev)
    g = torch.from_numpy(wl.g).to(dev)
    beta = _bf16(wl.beta, torch, dev)
    dO = _bf16(wl.d_out, torch, dev)
    scale = wl.scale
    out = torch.empty(v.shape, dtype=torch.bfloat16, device=dev)
    fs = torch.empty((B, H, K, V), dtype=torch.float32, device=dev)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    dg = torch.empty_like(g)
    db = torch.empty_like(beta)
    dS0 = torch.empty((B, H, K, V), dtype=torch.float32, device=dev)
    # training route: the forward keeps every chunk's start state and T tiles
    # (saved buffer), the backward reuses them
    ws_f_n = gdn.gdn_chunk_saved_size(B, T, H, K, V, 0)
    ws_b_n = gdn.gdn_chunk_bwd_saved_workspace_size(B, T, H, K, V, 0)
    ws_f = torch.empty(max(ws_f_n, 1), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(max(ws_b_n, 1), dtype=torch.uint8, device=dev)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def fwd():
        gdn.gdn_chunk_fwd_save(q, k, v, g, beta, scale, None, None, out, fs, B, T, H, K, V,
                               ws_f, ws_f_n, stream)

    def bwd():
        gdn.gdn_chunk_bwd_saved(q, k, v, g, beta, scale, None, dO, None, dq, dk, dv, dg, db,
                                dS0, B, T, H, K, V, ws_f, ws_f_n, ws_b, ws_b_n, stream)

    for _ in range(args.warmup):
        fwd()
        bwd()
    torch.cuda.synchronize()
    st = gdn.gdn_get_last_device_error()
    if st != 0:
        raise SystemExit(f"device error after warm-up: {gdn.gdn_status_string(st)}")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    launches0 = gdn.gdn_kernel_launches()
    t_wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()                    # evict L2 between steps (outside the events)
        ev[i][0].record(stream)
        fwd()
        ev[i][1].record(stream)
        bwd()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    launches = gdn.gdn_kernel_launches() - launches0
    barrier(world)
    clk = clocks.stop()
    st = gdn.gdn_get_last_device_error()
    if st != 0:
        raise SystemExit(f"device error in timed region: {gdn.gdn_status_string(st)}")

    t_fwd = statistics.mean(e[0].elapsed_time(e[1]) for e in ev) * 1e-3
    t_bwd = statistics.mean(e[1].elapsed_time(e[2]) for e in ev) * 1e-3
    t_step = max_over_ranks(t_fwd + t_bwd, world, dev)
    t_fwd_max = max_over_ranks(t_fwd, world, dev)
    t_bwd_max = max_over_ranks(t_bwd, world, dev)

    th, f_fwd, b_fwd, f_bwd, b_bwd = workload_totals(B, T, H, K, V)
    peaks, peaks_kind = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    tflops = float(peaks["bf16_tflops"])

    def roof(t, flops, nbytes):
        t_roof = max(flops / (tflops * 1e12), nbytes / (hbm * 1e9))
        bound = "hbm" if nbytes / (hbm * 1e9) >= flops / (tflops * 1e12) else "tensor"
        if bound == "hbm":
            ach = nbytes / t / 1e9
            return {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                    "frac": ach / hbm, "traffic": None, "roofline_us": t_roof * 1e6,
                    "measured_us": t * 1e6, "peak_source": peaks_kind}
        ach = flops / t / 1e12
        return {"bound": "tensor", "achieved": ach, "peak": tflops, "unit": "TFLOP/s",
                "frac": ach / tflops, "traffic": None, "roofline_us": t_roof * 1e6,
                "measured_us": t * 1e6, "peak_source": peaks_kind}

    roof_fwd = roof(t_fwd_max, f_fwd, b_fwd)
    roof_bwd = roof(t_bwd_max, f_bwd, b_bwd)
    traffic = load_traffic()
    if traffic is not None:
        roof_fwd["traffic"] = traffic

    # ---- end to end through the public API with pinned host buffers ----
    e2e = None
    if not args.no_e2e:
        barrier(world)
        e2e = measure_e2e(args, wl, dev, stream, gdn, torch, fs, dS0, ws_f, ws_f_n, ws_b, ws_b_n)
        t_e2e = max_over_ranks(e2e["ms_per_step"] * 1e-3, world, dev)
        e2e["ms_per_step"] = t_e2e * 1e3
        e2e["value"] = aggregate_rate(world, th, t_e2e)

    # ---- inference forward (gdn_chunk_fwd, nothing kept) on the same inputs ----
    t_inf = measure_inference_fwd(gdn, (q, k, v, g, beta, scale, out, fs), (B, T, H, K, V), flush,
                                  stream, torch, max(5, min(args.steps, 20)))
    t_inf = max_over_ranks(t_inf, world, dev)
    roof_inf = roof(t_inf, f_fwd, b_fwd)
    # ---- peak probes (our copy and tcgen05 GEMM kernels), in this run ----
    probes = None if args.no_probes else measure_probes(gdn, torch, dev, stream)
    if probes:
        for r in (roof_fwd, roof_bwd, roof_inf):
            if r["bound"] == "hbm":
                r["frac_of_probe"] = r["achieved"] / probes["copy_gbs"]
    # ---- sequence split on the long slow-decay workload ----
    split = None if args.no_decode else measure_split(gdn, torch, dev, stream)
    # ---- per-channel gate (KDA): chunked CUDA-core forward beside the token-serial one ----
    kda = None if args.no_decode else measure_kda(gdn, torch, dev, stream, clk)
    # ---- decode: the token-serial path, one token per call ----
    decode = None if args.no_decode else measure_decode(gdn, torch, dev, stream, hbm)
    # ---- prologue (q/k normalisation, gates) and its reverse mode at this shape ----
    prologue = None if args.no_decode else measure_prologue(gdn, torch, dev, stream, hbm, B * T, H, K)

    # ---- the other synthetic workloads: throughput, and accuracy on rank 0 at N = 1 ----
    configs = None
    if not args.no_configs:
        configs = measure_configs(gdn, torch, dev, stream, peaks,
                                  accuracy=(rank == 0 and world == 1 and not args.no_cpu_baseline))
    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N = 1) ----
    cpu = None
    accuracy = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import metrics, recurrence
        recurrence.build_oracle()
        threads = recurrence.default_threads()
        th_s, secs, done, fres, bres = oracle_sample(wl, args.cpu_seconds, threads)
        cpu = {"value": th_s / secs, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": (f"{len(done)} of {B * H} (batch, head) units at T={T}, fwd + reverse "
                          f"mode, fp64, {secs:.1f} s")}
        # accuracy of the timed GPU outputs on the sampled units
        o_gpu = bf16_np(out)
        grads = {n: bf16_np(t) for n, t in (("dq", dq), ("dk", dk), ("dv", dv), ("dbeta", db))}
        grads["dg"] = dg.cpu().numpy()
        rb = [s for (s, h) in done]
        rh = [h for (s, h) in done]
        accuracy = {"units": len(done),
                    "out_rel_rms": metrics.rel_l2(o_gpu[rb, :, rh], fres[0][rb, :, rh]),
                    "out_max_rel": metrics.max_rel(o_gpu[rb, :, rh], fres[0][rb, :, rh]),
                    "state_rel_rms": metrics.rel_l2(fs.cpu().numpy()[rb, rh], fres[1][rb, rh])}
        for n, x in grads.items():
            accuracy[f"{n}_rel_rms"] = metrics.rel_l2(x[rb, :, rh], bres[n][rb, :, rh])

    if rank == 0:
        line = {
            "metric": METRIC, "value": aggregate_rate(world, th, t_step), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": "dense fwd+bwd B=4 H=16 T=4096 d_k=128 d_v=128",
                       "global_batch": B * world, "seq_len": T, "heads": H, "d_k": K, "d_v": V,
                       "io": "bf16 q/k/v/beta/out/dO/grads, fp32 g and states",
                       "parallelism": f"dp{world} (independent batches, no collective)",
                       "l2": "flushed between steps (write of 2x L2) and inputs > L2"},
            "roofline": roof_fwd,
            "roofline_bwd": roof_bwd,
            "inference_fwd": {"tokens_heads_per_s": aggregate_rate(world, th, t_inf), "ms": t_inf * 1e3,
                              "roofline": roof_inf},
            "fwd": {"tokens_heads_per_s": aggregate_rate(world, th, t_fwd_max), "ms": t_fwd_max * 1e3},
            "bwd": {"tokens_heads_per_s": aggregate_rate(world, th, t_bwd_max), "ms": t_bwd_max * 1e3},
            "gpu_launches": int(launches),
            "wall_s_timed": t_wall,
            "clocks": clk,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "accuracy": accuracy,
            "probes": probes,
            "split": split,
            "kda": kda,
            "decode": decode,
            "prologue": prologue,
            "configs": configs,
        }
        print(json.dumps(line), flush=True)
    barrier(world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def bf16_np(t):
    import numpy as np
    import torch
    bits = t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def load_traffic():
    """DRAM traffic of one forward call (its launches summed) from the
    committed ncu summary, when it was taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    import hashlib
    csrc = os.path.join(ROOT, "linear_attention_sequence_chunked_gb300", "csrc")
    for name, digest in d.get("sources", {}).items():
        try:
            with open(os.path.join(csrc, name), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest() != digest:
                    return None
        except Exception:
            return None
    if not d.get("sources"):
        return None
    return d.get("bytes_per_launch")


def measure_inference_fwd(gdn, tensors, dims, flush, stream, torch, steps, warmup=3):
    """gdn_chunk_fwd alone (inference: output and final state, nothing kept
    for a backward) on the step's inputs, L2 flushed before each call;
    returns the mean duration in seconds."""
    q, k, v, g, beta, scale, out, fs = tensors
    B, T, H, K, V = dims
    n = gdn.gdn_chunk_fwd_workspace_size(B, T, H, K, V, 0)
    ws = torch.empty(max(n, 1), dtype=torch.uint8, device=q.device)

    def call():
        gdn.gdn_chunk_fwd(q, k, v, g, beta, scale, None, None, out, fs, B, T, H, K, V,
                          ws if n else None, n, stream)
    for _ in range(warmup):
        call()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    torch.cuda.synchronize()
    for e0, e1 in ev:
        flush.zero_()
        e0.record(stream)
        call()
        e1.record(stream)
    torch.cuda.synchronize()
    return statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev) * 1e-3


def measure_probes(gdn, torch, dev, stream, copy_bytes=2 << 30, n=8192, steps=10, warmup=3):
    """The peak probes in this run (our own kernels): a 2 GiB copy, counted
    as bytes read + bytes written, and an n x n by n x n bf16 GEMM on the
    tensor cores (2 n^3 FLOPs per call)."""
    src = torch.empty(copy_bytes, dtype=torch.uint8, device=dev).random_(0, 255)
    dst = torch.empty_like(src)

    def timed(call):
        for _ in range(warmup):
            call()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        torch.cuda.synchronize()
        for e0, e1 in ev:
            e0.record(stream)
            call()
            e1.record(stream)
        torch.cuda.synchronize()
        return statistics.median(e0.elapsed_time(e1) for e0, e1 in ev) * 1e-3

    t_copy = timed(lambda: gdn.gdn_probe_copy(src, dst, copy_bytes, stream))
    del src, dst
    g = torch.Generator(device=dev).manual_seed(11)
    A = torch.randn((n, n), device=dev, generator=g).to(torch.bfloat16)
    B = torch.randn((n, n), device=dev, generator=g).to(torch.bfloat16)
    C = torch.empty((n, n), device=dev, dtype=torch.bfloat16)
    t_gemm = timed(lambda: gdn.gdn_probe_gemm_bf16(A, B, C, n, n, n, stream))
    st = gdn.gdn_get_last_device_error()
    if st != 0:
        raise SystemExit(f"device error in the probes: {gdn.gdn_status_string(st)}")
    return {"copy_gbs": 2 * copy_bytes / t_copy / 1e9, "copy_bytes": copy_bytes,
            "bf16_gemm_tflops": 2.0 * n ** 3 / t_gemm / 1e12, "gemm": f"{n}x{n} by {n}x{n}, bf16, fp32 accumulate",
            "kernels": "gdn_probe_copy, gdn_probe_gemm_bf16 (tcgen05), median of "
                       f"{steps} after {warmup} warm-up"}


def measure_split(gdn, torch, dev, stream, T=65536, H=16, K=128, V=128, segs=(2, 4), steps=5, warmup=2):
    """The sequence split on the long slow-decay workload (one sequence,
    T = 65536, 16 heads: 32 chains unsplit): gdn_chunk_fwd against
    gdn_chunk_fwd_split at a few segment counts, L2 flushed before each call.
    Inputs follow that workload's recipe (q, v ~ N(0,1), k L2-normalised,
    g = -1e-3, beta = sigmoid(N(0,1) - 2)), drawn on the device."""
    gen = torch.Generator(device=dev).manual_seed(4)
    q = torch.randn((1, T, H, K), device=dev, generator=gen).to(torch.bfloat16)
    k = torch.nn.functional.normalize(torch.randn((1, T, H, K), device=dev, generator=gen), dim=-1).to(torch.bfloat16)
    v = torch.randn((1, T, H, V), device=dev, generator=gen).to(torch.bfloat16)
    g = torch.full((1, T, H), -1e-3, device=dev)
    beta = torch.sigmoid(torch.randn((1, T, H), device=dev, generator=gen) - 2.0).to(torch.bfloat16)
    out = torch.empty_like(v)
    fs = torch.empty((1, H, K, V), dtype=torch.float32, device=dev)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    scale = K ** -0.5

    def timed(call):
        for _ in range(warmup):
            call()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        torch.cuda.synchronize()
        for e0, e1 in ev:
            flush.zero_()
            e0.record(stream)
            call()
            e1.record(stream)
        torch.cuda.synchronize()
        return statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev) * 1e-3

    n = gdn.gdn_chunk_fwd_workspace_size(1, T, H, K, V, 0)
    ws = torch.empty(max(n, 1), dtype=torch.uint8, device=dev)
    t_u = timed(lambda: gdn.gdn_chunk_fwd(q, k, v, g, beta, scale, None, None, out, fs, 1, T, H, K, V,
                                          ws, n, stream))
    ref = out.float().clone()
    del ws
    res = {"config": f"1 sequence x T={T} x H={H}, d_k={K}, d_v={V}, g = -1e-3 (slow decay)",
           "unsplit_ms": t_u * 1e3, "unsplit_tokens_heads_per_s": T * H / t_u}
    for nseg in segs:
        n = gdn.gdn_chunk_fwd_split_workspace_size(1, T, H, K, V, nseg)
        ws = torch.empty(n, dtype=torch.uint8, device=dev)
        t_s = timed(lambda: gdn.gdn_chunk_fwd_split(q, k, v, g, beta, scale, None, out, fs, 1, T, H, K, V,
                                                    nseg, ws, n, stream))
        diff = float((out.float() - ref).norm() / ref.norm())
        res[f"nseg_{nseg}"] = {"ms": t_s * 1e3, "tokens_heads_per_s": T * H / t_s, "speedup": t_u / t_s,
                               "rel_l2_vs_unsplit": diff}
        del ws
    st = gdn.gdn_get_last_device_error()
    if st != 0:
        raise SystemExit(f"device error in the split measurement: {gdn.gdn_status_string(st)}")
    return res


FP32_LANES_PER_SM = 128   # fp32 FMA lanes per SM (4 sub-partitions x 32)
SMS = 152


def measure_kda(gdn, torch, dev, stream, clk, B=4, H=16, T=4096, K=128, V=128, steps=5, warmup=2, once=False):
    """The per-channel-gate (KDA) operator at the headline shape, L2 flushed
    before each call: the chunked forward through its workspace route (the
    chunk-parallel T/P kernel on the CUDA cores, then the tensor-core walk),
    the same forward without a workspace (fp32 CUDA-core walk), the
    token-serial forward, and the chunked backward (gdn_kda_chunk_bwd).
    Inputs: q, v, dO ~ N(0,1), k L2-normalised, g = -5 sigmoid(N(0,1) + 2) per
    key channel (the bounded gate with lower bound -5), beta = sigmoid(N(0,1)),
    zero initial state; drawn on the device.  With once, a profiling aid:
    one forward through the workspace route and one backward, untimed.  The
    roofline line is the
    forward's chunk-algebra FLOPs (decay exponentials not counted) against
    the fp32 FMA rate of 152 SMs x 128 lanes x 2 FLOP at the sampled SM
    clock: its dominant kernel, the T/P kernel, runs on the CUDA cores."""
    gen = torch.Generator(device=dev).manual_seed(5)
    q = torch.randn((B, T, H, K), device=dev, generator=gen).to(torch.bfloat16)
    k = torch.nn.functional.normalize(torch.randn((B, T, H, K), device=dev, generator=gen), dim=-1).to(torch.bfloat16)
    v = torch.randn((B, T, H, V), device=dev, generator=gen).to(torch.bfloat16)
    g = -5.0 * torch.sigmoid(torch.randn((B, T, H, K), device=dev, generator=gen) + 2.0)
    beta = torch.sigmoid(torch.randn((B, T, H), device=dev, generator=gen)).to(torch.bfloat16)
    d_out = torch.randn((B, T, H, V), device=dev, generator=gen).to(torch.bfloat16)
    out = torch.empty_like(v)
    fs = torch.empty((B, H, K, V), dtype=torch.float32, device=dev)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    scale = K ** -0.5
    nf = gdn.gdn_kda_chunk_fwd_workspace_size(B, T, H, K, V, 0)
    wf = torch.empty(nf, dtype=torch.uint8, device=dev)
    nb = gdn.gdn_kda_chunk_bwd_workspace_size(B, T, H, K, V, 0)
    wb = torch.empty(nb, dtype=torch.uint8, device=dev)
    grads = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(g),
             torch.empty_like(beta), torch.empty((B, H, K, V), dtype=torch.float32, device=dev)]

    def timed(fn, n):
        for _ in range(warmup):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        torch.cuda.synchronize()
        for e0, e1 in ev:
            flush.zero_()
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize()
        return statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev) * 1e-3

    def fwd(ws, nbytes, fn=gdn.gdn_kda_chunk_fwd):
        def run():
            if fn is gdn.gdn_kda_chunk_fwd:
                fn(q, k, v, g, beta, scale, None, None, out, fs, B, T, H, K, V, ws, nbytes, stream)
            else:
                fn(q, k, v, g, beta, scale, None, None, out, fs, B, T, H, K, V, stream)
        return run

    def bwd():
        gdn.gdn_kda_chunk_bwd(q, k, v, g, beta, scale, None, None, d_out, None, *grads, B, T, H, K, V, wb, nb, stream)

    if once:
        fwd(wf, nf)()
        bwd()
        torch.cuda.synchronize()
        st = gdn.gdn_get_last_device_error()
        if st != 0:
            raise SystemExit(f"device error in the KDA call: {gdn.gdn_status_string(st)}")
        return {"config": f"B={B} T={T} H={H} d_k={K} d_v={V}", "once": True}
    t_c = timed(fwd(wf, nf), steps)
    o_c = out.float().clone()
    t_w = timed(fwd(None, 0), 2)
    t_r = timed(fwd(None, 0, gdn.gdn_kda_recurrent_fwd), 2)
    diff = float((out.float() - o_c).norm() / out.float().norm())
    t_b = timed(bwd, steps)
    st = gdn.gdn_get_last_device_error()
    if st != 0:
        raise SystemExit(f"device error in the KDA measurement: {gdn.gdn_status_string(st)}")
    units = B * T * H
    mhz = (clk or {}).get("sm_mhz") or (clk or {}).get("sm_max_mhz") or 2070.0
    peak = SMS * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12
    ach = fwd_flops(K, V) * units / t_c / 1e12
    return {"config": f"B={B} T={T} H={H} d_k={K} d_v={V}, per-channel g in (-5, 0)",
            "chunk_ms": t_c * 1e3, "chunk_tokens_heads_per_s": units / t_c,
            "chunk_fp32_walk_ms": t_w * 1e3,
            "token_serial_ms": t_r * 1e3, "token_serial_tokens_heads_per_s": units / t_r,
            "speedup_vs_token_serial": t_r / t_c, "out_rel_l2_chunk_vs_token_serial": diff,
            "bwd_ms": t_b * 1e3, "fwd_bwd_tokens_heads_per_s": units / (t_c + t_b),
            "roofline": {"bound": "alu", "achieved": ach, "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
                         "peak_from": f"{SMS} SMs x {FP32_LANES_PER_SM} fp32 lanes x 2 FLOP x {mhz:.0f} MHz",
                         "traffic": None}}


def measure_decode(gdn, torch, dev, stream, hbm, B=256, H=16, K=128, V=128, steps=50, warmup=5):
    """gdn_recurrent_fwd one token per call, the state carried between two
    buffers (decode of B sequences).  Its bytes are dominated by the fp32
    state read and written per call: 8KV per (sequence, head) + the token's
    q, k, v, out (bf16), g (fp32), beta (bf16).  At B=256 each state buffer
    (256 MiB) exceeds L2, so every call reads its state from HBM."""
    import numpy as np
    rng = np.random.default_rng(7)
    q = torch.from_numpy(rng.standard_normal((B, 1, H, K), dtype=np.float32)).to(dev).to(torch.bfloat16)
    k = torch.nn.functional.normalize(torch.from_numpy(
        rng.standard_normal((B, 1, H, K), dtype=np.float32)).to(dev), dim=-1).to(torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((B, 1, H, V), dtype=np.float32)).to(dev).to(torch.bfloat16)
    g = torch.full((B, 1, H), -0.05, dtype=torch.float32, device=dev)
    beta = torch.full((B, 1, H), 0.5, dtype=torch.bfloat16, device=dev)
    out = torch.empty((B, 1, H, V), dtype=torch.bfloat16, device=dev)
    st = [torch.zeros((B, H, K, V), dtype=torch.float32, device=dev) for _ in range(2)]
    scale = K ** -0.5
    for i in range(warmup):
        gdn.gdn_recurrent_fwd(q, k, v, g, beta, scale, st[i & 1], None, out, st[1 - (i & 1)],
                              B, 1, H, K, V, stream)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(steps):
        gdn.gdn_recurrent_fwd(q, k, v, g, beta, scale, st[i & 1], None, out, st[1 - (i & 1)],
                              B, 1, H, K, V, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) * 1e-3 / steps
    nbytes = B * H * (8 * K * V + 2 * (2 * K + 2 * V) + 4 + 2)
    return {"config": f"B={B} sequences x H={H}, d_k={K}, d_v={V}, one token per call",
            "value": B * H / t, "unit": UNIT, "us_per_call": t * 1e6,
            "roofline": {"bound": "hbm", "achieved": nbytes / t / 1e9, "peak": hbm, "unit": "GB/s",
                         "frac": nbytes / t / 1e9 / hbm}}


def measure_prologue(gdn, torch, dev, stream, hbm, rows, H, K, steps=20, warmup=3):
    """gdn_prologue_fwd and gdn_prologue_bwd (decay gate, beta factor 2) on
    rows x H (token, head) rows; HBM-bound, algorithmic bytes: forward reads
    q, k and writes their normalised copies (bf16) plus the gates; backward
    reads q, k and the two gradients and writes dq, dk (bf16) plus the gate
    gradients."""
    gen = torch.Generator(device=dev).manual_seed(5)
    q = torch.randn((rows, H, K), device=dev, generator=gen).to(torch.bfloat16)
    k = torch.randn((rows, H, K), device=dev, generator=gen).to(torch.bfloat16)
    a = torch.randn((rows, H), device=dev, generator=gen)
    b = torch.randn((rows, H), device=dev, generator=gen)
    A_log = torch.rand((H,), device=dev, generator=gen)
    dtb = torch.rand((H,), device=dev, generator=gen) - 0.5
    qo, ko = torch.empty_like(q), torch.empty_like(k)
    g = torch.empty((rows, H), device=dev)
    beta = torch.empty((rows, H), device=dev, dtype=torch.bfloat16)
    dq = torch.randn((rows, H, K), device=dev, generator=gen).to(torch.bfloat16)
    dk = torch.randn((rows, H, K), device=dev, generator=gen).to(torch.bfloat16)
    dg = torch.randn((rows, H), device=dev, generator=gen)
    dbeta = torch.randn((rows, H), device=dev, generator=gen).to(torch.bfloat16)
    dqr, dkr = torch.empty_like(q), torch.empty_like(k)
    da, db = torch.empty_like(a), torch.empty_like(b)
    dA, ddt = torch.empty_like(A_log), torch.empty_like(dtb)

    def fwd():
        gdn.gdn_prologue_fwd(q, k, a, b, A_log, dtb, 1, -5.0, 2.0, qo, ko, g, beta, rows, H, K, stream)

    def bwd():
        gdn.gdn_prologue_bwd(q, k, a, b, A_log, dtb, 1, -5.0, 2.0, dq, dk, dg, dbeta, dqr, dkr,
                             da, db, dA, ddt, rows, H, K, stream)

    res = {}
    n = rows * H
    for name, fn, nbytes in (("fwd", fwd, n * (8 * K + 4 + 4 + 4 + 2)),
                             ("bwd", bwd, n * (12 * K + 4 + 4 + 4 + 2 + 4 + 4))):
        for _ in range(warmup):
            fn()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) * 1e-3 / steps
        res[name] = {"us": t * 1e6, "achieved_gbs": nbytes / t / 1e9, "frac": nbytes / t / 1e9 / hbm}
    res["config"] = f"{rows} tokens x H={H}, d_k={K}, decay gate, beta factor 2"
    return res


def _dev_inputs(wl, torch, dev):
    d = dict(q=_bf16(wl.q, torch, dev), k=_bf16(wl.k, torch, dev), v=_bf16(wl.v, torch, dev),
             g=torch.from_numpy(wl.g).to(dev), beta=_bf16(wl.beta, torch, dev))
    d["cu"] = None if wl.cu_seqlens is None else torch.from_numpy(wl.cu_seqlens).to(dev)
    d["dO"] = None if wl.d_out is None else _bf16(wl.d_out, torch, dev)
    return d


def _timed(call, torch, stream, flush, steps, warmup=3):
    for _ in range(warmup):
        call()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    for e0, e1 in ev:
        flush.zero_()
        e0.record(stream)
        call()
        e1.record(stream)
    torch.cuda.synchronize()
    return statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev) * 1e-3


def measure_configs(gdn, torch, dev, stream, peaks, accuracy, steps=10):
    """Throughput and accuracy on the other synthetic workloads, beside the
    headline step:
      * correlated varlen (2 x 5120 packed, H=12, d=128, bounded gates;
        fla issue #1550's CP2 inputs): inference forward, out/state rel-RMS
        over all 24 (sequence, head) units;
      * slow decay (B=1, T=65536, H=16, d=128, g = -1e-3; cuLA issue #126's
        64K heads): inference forward, per-head rel-L2 in 8 windows of 8192
        tokens, all 16 heads;
      * training shape (B=8, T=4096, H=16, d_k=128, d_v=256, beta in (0,2)):
        the training step (forward keeping states + backward from them),
        out/state/gradient rel-RMS on heads 0 and 15 of batch 0;
      * the dense sweep's d_k = 64 rows at T=4096 ((64,64), (64,128)):
        inference forward, out/state rel-RMS on three units.
    Each call is timed with CUDA events after 3 warm-up calls, L2 flushed
    before each call.  With `accuracy` (rank 0, one GPU) the fp64 oracle is
    run on the units named above and compared with the timed call's
    results."""
    import numpy as np
    from linear_attention_sequence_chunked_gb300 import workloads as W
    hbm = float(peaks["hbm_gbs"])
    tflops = float(peaks["bf16_tflops"])
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    res = {}

    def roof(t, flops, nbytes):
        bound = "hbm" if nbytes / (hbm * 1e9) >= flops / (tflops * 1e12) else "tensor"
        if bound == "hbm":
            ach = nbytes / t / 1e9
            return {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm}
        ach = flops / t / 1e12
        return {"bound": "tensor", "achieved": ach, "peak": tflops, "unit": "TFLOP/s", "frac": ach / tflops}

    def fwd_case(name, wl, units, windows=False):
        d = _dev_inputs(wl, torch, dev)
        N, T, H, K, V = wl.n_seq, wl.T, wl.H, wl.d_k, wl.d_v
        varlen = wl.cu_seqlens is not None
        out = torch.empty(d["v"].shape, dtype=torch.bfloat16, device=dev)
        fs = torch.empty((N, H, K, V), dtype=torch.float32, device=dev)
        n = gdn.gdn_chunk_fwd_workspace_size(N, T, H, K, V, varlen)
        ws = torch.empty(max(n, 1), dtype=torch.uint8, device=dev)
        t = _timed(lambda: gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], wl.scale, None,
                                             d["cu"], out, fs, N, T, H, K, V, ws, n, stream),
                   torch, stream, flush, steps)
        st = gdn.gdn_get_last_device_error()
        if st != 0:
            raise SystemExit(f"device error in {name}: {gdn.gdn_status_string(st)}")
        th = wl.token_heads
        r = {"ms": t * 1e3, "tokens_heads_per_s": th / t,
             "roofline": roof(t, fwd_flops(K, V) * th, fwd_bytes(K, V) * th + 4 * K * V * N * H)}
        if accuracy:
            from oracle import metrics, recurrence
            o_ref, S_ref = recurrence.workload_fwd(wl, units=units)
            o = bf16_np(out)
            S = fs.cpu().numpy()
            per = []
            for (s_, h_) in units:
                b_, t0, t1 = wl.seq_bounds()[s_]
                e = {"unit": [s_, h_], "out_rel_rms": metrics.rel_l2(o[b_, t0:t1, h_], o_ref[b_, t0:t1, h_]),
                     "state_rel_rms": metrics.rel_l2(S[s_, h_], S_ref[s_, h_])}
                if windows:
                    e["window_rel_l2"] = metrics.window_rel_l2(o[b_, t0:t1, h_], o_ref[b_, t0:t1, h_], axis=0)
                per.append(e)
            acc = {"units": len(units),
                   "out_rel_rms_max": max(e["out_rel_rms"] for e in per),
                   "state_rel_rms_max": max(e["state_rel_rms"] for e in per)}
            if not windows:
                sel = [(wl.seq_bounds()[s_], h_) for (s_, h_) in units]
                acc["out_rel_rms_all"] = metrics.rel_l2(
                    np.concatenate([o[b_, t0:t1, h_].ravel() for (b_, t0, t1), h_ in sel]),
                    np.concatenate([o_ref[b_, t0:t1, h_].ravel() for (b_, t0, t1), h_ in sel]))
            else:
                acc["window_rel_l2_max"] = max(max(e["window_rel_l2"]) for e in per)
                acc["window_rel_l2_per_head"] = [[round(x, 7) for x in e["window_rel_l2"]] for e in per]
            r["accuracy"] = acc
        return r

    wl3 = W.make_workload(3)
    res["correlated_varlen"] = fwd_case("correlated varlen", wl3,
                                        [(s_, h_) for s_ in range(wl3.n_seq) for h_ in range(wl3.H)])
    res["correlated_varlen"]["config"] = "2 x 5120 packed, H=12, d_k=d_v=128, correlated q/k, g = -5 sigmoid(N)"
    if accuracy:
        res["correlated_varlen"]["accuracy"]["pages_context"] = (
            "fla ordinary chunk kernel 1.3509 % rel-RMS on its CP2 inputs (fla issue #1550); threshold 0.008")
    del wl3
    wl4 = W.make_workload(4)
    res["slow_decay"] = fwd_case("slow decay", wl4, [(0, h_) for h_ in range(wl4.H)], windows=True)
    res["slow_decay"]["config"] = "B=1 T=65536 H=16 d_k=d_v=128, g = -1e-3, 8 windows of 8192 tokens"
    if accuracy:
        res["slow_decay"]["accuracy"]["pages_context"] = (
            "cuLA intracard split on H200: windows 1-7 at about 7.3e-3 rel-L2 (cuLA issue #126)")
    del wl4
    for (dk, dv) in ((64, 64), (64, 128)):
        wl2 = W.make_workload(2, d_k=dk, d_v=dv)
        key = f"dense_dk{dk}_dv{dv}"
        res[key] = fwd_case(key, wl2, [(0, 0), (1, 7), (3, 15)])
        res[key]["config"] = f"B=4 T=4096 H=16 d_k={dk} d_v={dv}"
        del wl2

    # training shape: the training step
    wl5 = W.make_workload(5, with_grad=True)
    d = _dev_inputs(wl5, torch, dev)
    B, T, H, K, V = wl5.B, wl5.T, wl5.H, wl5.d_k, wl5.d_v
    out = torch.empty(d["v"].shape, dtype=torch.bfloat16, device=dev)
    fs = torch.empty((B, H, K, V), dtype=torch.float32, device=dev)
    grads = dict(dq=torch.empty_like(d["q"]), dk=torch.empty_like(d["k"]), dv=torch.empty_like(d["v"]),
                 dg=torch.empty_like(d["g"]), dbeta=torch.empty_like(d["beta"]),
                 dS0=torch.empty((B, H, K, V), dtype=torch.float32, device=dev))
    nf = gdn.gdn_chunk_saved_size(B, T, H, K, V, 0)
    nb = gdn.gdn_chunk_bwd_saved_workspace_size(B, T, H, K, V, 0)
    ws_f = torch.empty(nf, dtype=torch.uint8, device=dev)
    ws_b = torch.empty(max(nb, 1), dtype=torch.uint8, device=dev)

    def fwd():
        gdn.gdn_chunk_fwd_save(d["q"], d["k"], d["v"], d["g"], d["beta"], wl5.scale, None, None, out, fs,
                               B, T, H, K, V, ws_f, nf, stream)

    def bwd():
        gdn.gdn_chunk_bwd_saved(d["q"], d["k"], d["v"], d["g"], d["beta"], wl5.scale, None, d["dO"], None,
                                grads["dq"], grads["dk"], grads["dv"], grads["dg"], grads["dbeta"],
                                grads["dS0"], B, T, H, K, V, ws_f, nf, ws_b, nb, stream)
    t_f = _timed(fwd, torch, stream, flush, steps)
    t_b = _timed(lambda: (fwd(), bwd()), torch, stream, flush, steps) - t_f
    st = gdn.gdn_get_last_device_error()
    if st != 0:
        raise SystemExit(f"device error in the training shape: {gdn.gdn_status_string(st)}")
    th = wl5.token_heads
    r = {"config": "B=8 T=4096 H=16 d_k=128 d_v=256, beta in (0,2): forward keeping states + backward",
         "step_ms": (t_f + t_b) * 1e3, "tokens_heads_per_s": th / (t_f + t_b),
         "fwd_ms": t_f * 1e3, "bwd_ms": t_b * 1e3,
         "roofline_fwd": roof(t_f, fwd_flops(K, V) * th, fwd_bytes(K, V) * th + 4 * K * V * B * H),
         "roofline_bwd": roof(t_b, bwd_flops(K, V) * th, bwd_bytes(K, V) * th)}
    if accuracy:
        from oracle import metrics, recurrence
        units = [(0, 0), (0, 15)]
        o_ref, S_ref = recurrence.workload_fwd(wl5, units=units)
        g_ref = recurrence.workload_bwd(wl5, units=units)
        o = bf16_np(out)
        S = fs.cpu().numpy()
        gg = {n_: (bf16_np(x) if x.dtype == torch.bfloat16 else x.cpu().numpy()) for n_, x in grads.items()}
        acc = {"units": units}
        for (s_, h_) in units:
            e = {"out": metrics.rel_l2(o[s_, :, h_], o_ref[s_, :, h_]),
                 "state": metrics.rel_l2(S[s_, h_], S_ref[s_, h_])}
            for n_ in ("dq", "dk", "dv", "dg", "dbeta"):
                e[n_] = metrics.rel_l2(gg[n_][s_, :, h_], g_ref[n_][s_, :, h_])
            e["dS0"] = metrics.rel_l2(gg["dS0"][s_, h_], g_ref["dS0"][s_, h_])
            acc[f"rel_rms_b{s_}_h{h_}"] = e
        r["accuracy"] = acc
    res["training_shape"] = r
    return res


def measure_e2e(args, wl, dev, stream, gdn, torch, fs, dS0, ws_f, ws_f_n, ws_b, ws_b_n):
    """The step through the public API with host buffers: every step copies
    its inputs in from pinned host memory and its outputs and gradients back,
    all inside the timed region.  A step's inputs sit in one pinned host
    block and its results in one device block (each tensor a 256-byte
    aligned view), so each direction is one copy per step (the results two:
    the forward's as soon as the forward ends, the gradients after the
    backward).  Steps are
    pipelined the way a prefetching loader runs them: step i + 1's inputs go
    in (copy stream) and step i - 1's results come out (a second copy stream)
    while step i computes; device blocks alternate between two sets, ordered
    by events (a third set, letting the input copies run further ahead,
    measured slower)."""
    import numpy as np
    B, T, H, K, V = wl.B, wl.T, wl.H, wl.d_k, wl.d_v
    in_specs = [("q", (B, T, H, K), torch.int16), ("k", (B, T, H, K), torch.int16),
                ("v", (B, T, H, V), torch.int16), ("g", (B, T, H), torch.float32),
                ("beta", (B, T, H), torch.int16), ("dO", (B, T, H, V), torch.int16)]
    # the forward's results first: they start back while the backward runs
    out_specs = [("out", (B, T, H, V), torch.int16), ("fs", tuple(fs.shape), torch.float32),
                 ("dq", (B, T, H, K), torch.int16), ("dk", (B, T, H, K), torch.int16),
                 ("dv", (B, T, H, V), torch.int16), ("dg", (B, T, H), torch.float32),
                 ("dbeta", (B, T, H), torch.int16), ("dS0", tuple(dS0.shape), torch.float32)]

    def layout(specs):
        offs, off = {}, 0
        for n, shp, dt in specs:
            nbytes = int(np.prod(shp)) * torch.empty((), dtype=dt).element_size()
            offs[n] = (off, nbytes, shp, dt)
            off = (off + nbytes + 255) // 256 * 256
        return offs, off

    def views(block, offs):
        return {n: block[o:o + nb].view(dt).view(shp) for n, (o, nb, shp, dt) in offs.items()}

    in_offs, in_bytes = layout(in_specs)
    out_offs, out_bytes = layout(out_specs)
    h_in_blk = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    h_out_blk = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()
    h_in = views(h_in_blk, in_offs)
    src = {"q": wl.q, "k": wl.k, "v": wl.v, "g": wl.g, "beta": wl.beta, "dO": wl.d_out}
    for n, a in src.items():
        a = np.ascontiguousarray(a)
        h_in[n].copy_(torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a))
    nbuf = 2
    d_in_blk = [torch.empty(in_bytes, dtype=torch.uint8, device=dev) for _ in range(nbuf)]
    d_out_blk = [torch.empty(out_bytes, dtype=torch.uint8, device=dev) for _ in range(nbuf)]
    d_in = [views(x, in_offs) for x in d_in_blk]
    d_out = [views(x, out_offs) for x in d_out_blk]
    bf = lambda t: t.view(torch.bfloat16)  # noqa: E731
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731

    fwd_bytes = out_offs["dq"][0]  # out and the final state

    def run(n_steps):
        in_ready = [ev() for _ in range(n_steps)]
        fwd_done = [ev() for _ in range(n_steps)]
        comp_done = [ev() for _ in range(n_steps)]
        out_done = [ev() for _ in range(n_steps)]
        for i in range(n_steps):
            j = i % nbuf
            with torch.cuda.stream(s_in):
                if i >= nbuf:
                    s_in.wait_event(comp_done[i - nbuf])   # set j's inputs are free
                d_in_blk[j].copy_(h_in_blk, non_blocking=True)
                in_ready[i].record(s_in)
            stream.wait_event(in_ready[i])
            if i >= nbuf:
                stream.wait_event(out_done[i - nbuf])      # set j's outputs were read out
            di, do = d_in[j], d_out[j]
            gdn.gdn_chunk_fwd_save(bf(di["q"]), bf(di["k"]), bf(di["v"]), di["g"], bf(di["beta"]),
                                   wl.scale, None, None, bf(do["out"]), do["fs"], B, T, H, K, V,
                                   ws_f, ws_f_n, stream)
            fwd_done[i].record(stream)
            gdn.gdn_chunk_bwd_saved(bf(di["q"]), bf(di["k"]), bf(di["v"]), di["g"], bf(di["beta"]),
                                    wl.scale, None, bf(di["dO"]), None, bf(do["dq"]), bf(do["dk"]),
                                    bf(do["dv"]), do["dg"], bf(do["dbeta"]), do["dS0"], B, T, H, K, V,
                                    ws_f, ws_f_n, ws_b, ws_b_n, stream)
            comp_done[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(fwd_done[i])
                h_out_blk[:fwd_bytes].copy_(d_out_blk[j][:fwd_bytes], non_blocking=True)
                s_out.wait_event(comp_done[i])
                h_out_blk[fwd_bytes:].copy_(d_out_blk[j][fwd_bytes:], non_blocking=True)
                out_done[i].record(s_out)
        return out_done[-1]

    reps = max(4, min(args.steps, 12))
    run(nbuf)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    last = run(reps)
    s_out.wait_event(last)
    e1.record(s_out)
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) * 1e-3 / reps
    # the results that came back are the step's: the last output block holds them
    h_out = views(h_out_blk, out_offs)
    if not torch.isfinite(h_out["dS0"]).all():
        raise SystemExit("e2e: non-finite results read back")
    return {"value": B * T * H / t, "unit": UNIT, "h2d_bytes_per_step": int(in_bytes),
            "d2h_bytes_per_step": int(out_bytes), "ms_per_step": t * 1e3, "steps": reps,
            "pipelined": "copies of the neighbouring steps overlap each step's compute; inputs one copy, "
                         "results two (forward outputs while the backward runs, then the gradients)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-probes", action="store_true")
    ap.add_argument("--no-configs", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--split-only", type=int, default=0, metavar="NSEG",
                    help="run only the sequence-split measurement at NSEG segments (profiling)")
    ap.add_argument("--kda-once", default="", metavar="B,H,T",
                    help="run one per-channel-gate forward and backward at B,H,T (profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
