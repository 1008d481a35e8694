"""Benchmark of the KDA hot path on one GB300 (or N, one process per GPU).

One step = the whole path over one batch of the varlen workload: a packed
prefill of 64 sequences (lengths uniform in [128, 8192], H = 16, d_k = 128,
d_v = 256, chunk 64, bf16 q/k/v, fp32 alpha/beta/state) through kda_prefill
(planner + chunkwise kernel), then 32 kda_decode_step calls continuing every
sequence from its returned state.  Inputs are seeded synthetic data, resident
in HBM before timing; they exceed L2 (about 11 GB per step), so no flush is
needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 CPU
oracle on the host cores instead, on a bounded sample of the same workload.
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
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from gated_delta_rule_45_gb300 import synth  # noqa: E402

METRIC = "KDA prefill tokens/s & decode state-updates/s at 1 GB300; % of TC/HBM roofline"
UNIT = "tokens/s"

# DRAM traffic of one launch of the dominant kernel (the tensor-core prefill on
# this workload's full-size batch), from a 1-pass ncu capture of
# dram__bytes_read.sum + dram__bytes_write.sum.  It is reported only while the
# kernel's source is the one the capture was taken on (its sha256 below);
# after any change to the kernel it is null until captured again.
TRAFFIC_CAPTURE = {
    "bytes_per_launch": 10.33e9,
    "date": "2026-12-03",
    "sources_sha256": "653da9a9b41098d5e235e629e375cb1736a2786ef3cbbd276fed685b1654a904",
}
TRAFFIC_SOURCES = ("gated_delta_rule_45_gb300/csrc/kda_prefill_tc.cu",
                   "gated_delta_rule_45_gb300/csrc/kda_tc.cuh")


def kernel_sources_sha256() -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def stored_traffic():
    """(bytes per launch or None, where the figure comes from)."""
    cap = TRAFFIC_CAPTURE
    if cap["sources_sha256"] and cap["sources_sha256"] == kernel_sources_sha256():
        return cap["bytes_per_launch"], ("ncu capture of this kernel version (" + cap["date"]
                                         + "), dram__bytes_read.sum + dram__bytes_write.sum")
    return None, "no ncu capture of the current kernel version"


# ---------------------------------------------------------------- distributed
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(backend: str):
    ws, rank, _ = dist_env()
    if ws > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend=backend, rank=rank, world_size=ws)


def barrier():
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()


def reduce_max_sum(elapsed_s: float, units: float, device=None):
    """Max of elapsed time and sum of units over ranks (identity when single-process)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return elapsed_s, units
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    torch.distributed.all_reduce(u, op=torch.distributed.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi during the timed region."""
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- workload
def workload_bytes(spec, T: int, decode_steps: int, alpha_bytes: int | None = None):
    """Algorithmic HBM bytes of one prefill launch and of one decode step
    (alpha_bytes: bytes of the forget gate per token-head, fp32 per channel
    by default)."""
    esz = 2 if spec.dtype == "bf16" else 4
    if alpha_bytes is None:
        alpha_bytes = spec.d_v * 4
    per_token_head = 2 * spec.d_k * esz + spec.d_v * esz + alpha_bytes + 4 + spec.d_v * esz
    state = spec.num_seqs * spec.H * spec.d_v * spec.d_k * 4
    prefill = T * spec.H * per_token_head + 2 * state + 4 * (spec.num_seqs + 1)
    bh = spec.num_seqs * spec.H
    decode = bh * (2 * spec.d_k * esz + spec.d_v * esz + spec.d_v * 4 + 4 + spec.d_v * esz) \
        + 2 * state
    return prefill, decode


def make_workload(seed: int):
    spec = synth.VARLEN
    if seed != spec.seed:
        import dataclasses
        spec = dataclasses.replace(spec, seed=seed)
    d = synth.prefill_inputs(spec)
    steps = synth.decode_sequence_inputs(synth.VARLEN_DECODE_STEPS, spec.num_seqs, spec.H,
                                         spec.d_k, spec.d_v, spec.dtype, spec.alpha_mu,
                                         d["generator"])
    return spec, d, steps


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def bf16_peak():
    """Dense bf16 tensor peak (TFLOP/s) for a kernel timed alone (burst figure)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (burst)"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


# tcgen05 MMA flops the chunk kernel issues per (128-channel block, 64-token chunk):
# S[K;Q]^T 2 x 2x128x128x128 (hi, lo), [K;Q]K^T 2x128x64x128, U^T 3 x 2x128x64x64,
# S += U^T K 2 x 2x128x128x64, O^T += U^T P^T 3 x 2x128x64x64.
MMA_FLOPS_PER_BLOCK_CHUNK = (2 * 2 * 128 * 128 * 128 + 2 * 128 * 64 * 128
                             + 3 * 2 * 128 * 64 * 64 + 2 * 2 * 128 * 128 * 64
                             + 3 * 2 * 128 * 64 * 64)


# Algorithmic flops of the chunk form per token-head (d_k = d_v = 128, C = 64),
# every contraction counted as dense tiles: 4 C d_k + 4 C d_v + 6 d_k d_v; and
# counting only the causal triangles that carry work: 2 C d_k + 2 C d_v + 6 d_k d_v.
ALG_FLOPS_PER_TOKEN_HEAD = 4 * 64 * 128 + 4 * 64 * 128 + 6 * 128 * 128
ALG_FLOPS_PER_TOKEN_HEAD_USEFUL = 2 * 64 * 128 + 2 * 64 * 128 + 6 * 128 * 128


# Multiply-adds of the chunkwise backward per (64-value-row block, 64-token
# chunk), d_k = 128, each product counted once: the forward sweep (K K^T, Y,
# U, S update: 1,835,008) and the backward sweep (K K^T, Q K^T, Y, U, E, dU,
# dT, dX, dT T^T, dA, dM, dq, dk, D: 9,437,184).
BWD_FMA_PER_BLOCK_CHUNK = 1_835_008 + 9_437_184
# The same products as the kernel issues them on the tensor cores: a product
# with one hi/lo-split operand runs twice, with two split operands three
# times (forward sweep 3,407,872, backward sweep 21,495,808).
BWD_MMA_FMA_PER_BLOCK_CHUNK = 3_407_872 + 21_495_808


# ---------------------------------------------------------------- CPU oracle
def time_oracle_sample(d, steps, pairs_wanted: int, budget_s: float, seed: int = 0,
                       threads: int | None = None):
    """Time the oracle on sampled (sequence, head) pairs of the workload (prefill
    over the whole sequence, then the 32 decode tokens), on ``threads`` threads
    (default: every host core this process may use).  Returns (tokens/s, cores,
    description, seconds).  A token is counted per head, divided by H to give
    tokens (all heads) per second, the unit of the GPU figure."""
    import oracle
    spec = d["spec"]
    rng = np.random.default_rng(seed)
    cu = d["cu_seqlens"].numpy()
    cores = threads or (len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
                        else os.cpu_count())
    order = rng.permutation(spec.num_seqs * spec.H)
    chosen = []
    token_heads = 0
    # pick pairs until about the budget's worth of work (≈ 8 d_k d_v flop per token-head,
    # ~3.5 Gflop/s per core fp64 for this loop nest)
    per_core_rate = 3.5e9
    target = budget_s * per_core_rate * cores / (8.0 * spec.d_k * spec.d_v)
    for idx in order[:pairs_wanted]:
        n, h = divmod(int(idx), spec.H)
        chosen.append((n, h))
        token_heads += int(cu[n + 1] - cu[n]) + len(steps)
        if token_heads >= target:
            break
    # gather packed inputs: prefill tokens followed by the decode tokens of each pair
    qs, ks, vs, als, bes, lens, s0s = [], [], [], [], [], [], []
    for n, h in chosen:
        a, b = int(cu[n]), int(cu[n + 1])
        qs.append(torch.cat([d["q"][a:b, h]] + [st["q"][n, h][None] for st in steps]))
        ks.append(torch.cat([d["k"][a:b, h]] + [st["k"][n, h][None] for st in steps]))
        vs.append(torch.cat([d["v"][a:b, h]] + [st["v"][n, h][None] for st in steps]))
        als.append(torch.cat([d["alpha"][a:b, h]] + [st["alpha"][n, h][None] for st in steps]))
        bes.append(torch.cat([d["beta"][a:b, h]] + [st["beta"][n, h][None] for st in steps]))
        lens.append(b - a + len(steps))
        s0s.append(d["S0"][n, h].double().numpy())
    q = synth.bf16_bits(torch.cat(qs)[:, None])
    k = synth.bf16_bits(torch.cat(ks)[:, None])
    v = synth.bf16_bits(torch.cat(vs)[:, None])
    al = torch.cat(als)[:, None].numpy()
    be = torch.cat(bes)[:, None].numpy()
    pcu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    S0 = np.stack(s0s)[:, None]
    t0 = time.perf_counter()
    oracle.prefill(q, k, v, al, be, S0, pcu, nthreads=cores)
    dt = time.perf_counter() - t0
    th = int(pcu[-1])
    desc = (f"{len(chosen)} (sequence, head) pairs of the varlen workload, each over its "
            f"whole prefill plus its 32 decode tokens: {th} token-heads, fp64, "
            f"{dt:.1f} s on {cores} thread{'s' if cores != 1 else ''}; "
            f"tokens/s = token-heads/s / H")
    return th / dt / spec.H, cores, desc, dt


def time_oracle_backward_sample(d, dO, dS_T, budget_s: float, seed: int = 0):
    """Time the oracle's reverse mode on sampled (sequence, head) pairs of a
    prefill workload, one pair per host thread, each over its whole sequence.
    Returns (tokens/s, cores, description); tokens/s = token-heads/s / H."""
    import oracle
    spec = d["spec"]
    cu = d["cu_seqlens"].numpy()
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    rng = np.random.default_rng(seed)
    # about 40 d_k d_v fp64 flops per token-head (forward re-run + reverse), ~1.5 Gflop/s a core
    per_pair_s = 40.0 * spec.d_k * spec.d_v * float(np.mean(np.diff(cu))) / 1.5e9
    n_pairs = int(max(1, min(cores * max(1, round(budget_s / max(per_pair_s, 1e-3))),
                             spec.num_seqs * spec.H)))
    chosen = [divmod(int(i), spec.H) for i in rng.permutation(spec.num_seqs * spec.H)[:n_pairs]]
    parts = {key: [] for key in ("q", "k", "v", "alpha", "beta")}
    dos, lens = [], []
    for n, h in chosen:
        a, b = int(cu[n]), int(cu[n + 1])
        for key in parts:
            parts[key].append(d[key][a:b, h:h + 1])
        dos.append(dO[a:b, h:h + 1])
        lens.append(b - a)
    cat = lambda key: torch.cat(parts[key])
    pcu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    st = (len(chosen), 1, spec.d_v, spec.d_k)
    S0 = np.zeros(st) if d["S0"] is None else np.stack(
        [d["S0"][n, h].double().numpy() for n, h in chosen])[:, None]
    dst = np.stack([dS_T[n, h].double().numpy() for n, h in chosen])[:, None]
    t0 = time.perf_counter()
    oracle.backward(synth.bf16_bits(cat("q")), synth.bf16_bits(cat("k")), synth.bf16_bits(cat("v")),
                    cat("alpha").numpy(), cat("beta").numpy(), S0, pcu,
                    torch.cat(dos).double().numpy(), dst, nthreads=cores)
    dt = time.perf_counter() - t0
    th = int(pcu[-1])
    desc = (f"{len(chosen)} (sequence, head) pairs of the workload, reverse mode over each "
            f"whole sequence: {th} token-heads, fp64, {dt:.1f} s on {cores} threads; "
            f"tokens/s = token-heads/s / H")
    return th / dt / spec.H, cores, desc


def time_oracle_attnres_sample(x, calls, budget_s: float):
    """Time the Attention Residuals oracle (numpy fp64) on the first tokens of
    the network, every layer in turn with the stored block sums and the running
    sum carried as a model does.  Returns (tokens/s, cores, description)."""
    from oracle import attnres as ar
    spec = x["spec"]
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    scale = 1.0 / np.sqrt(spec.d)
    n_tok = 64
    max_tok = 1024   # keeps the fp64 copy of the layer outputs near 1 GB
    while True:
        h0 = x["h0"][:n_tok].cpu().double().numpy()
        outs = x["outs"][:, :n_tok].cpu().double().numpy()
        qs = x["queries"].cpu().double().numpy()
        t0 = time.perf_counter()
        blocks, partial, layer = [h0], None, 0
        h_last = None
        for n, size in enumerate(spec.block_sizes, start=1):
            for i in range(size):
                if i == 0 and n > 1:
                    _, P = ar.layer_step(np.stack(blocks), partial, h_last, qs[layer], scale)
                    blocks.append(P)
                    partial = None
                else:
                    _, partial = ar.layer_step(np.stack(blocks), partial, h_last, qs[layer],
                                               scale)
                h_last = outs[layer]
                layer += 1
        dt = time.perf_counter() - t0
        if dt >= 0.5 * budget_s or n_tok >= min(spec.T, max_tok):
            break
        n_tok = min(spec.T, max_tok, n_tok * max(2, int(budget_s / max(dt, 1e-3))))
    desc = (f"the first {n_tok} tokens through all {layer} layers, numpy fp64 "
            f"({dt:.1f} s; numpy's threads, up to {cores} cores)")
    return n_tok / dt, cores, desc


def run_reference(args):
    ws, rank, _ = dist_env()
    if ws > 1:
        init_dist("gloo")
        if rank != 0:
            barrier()
            return
    spec, d, steps = make_workload(synth.VARLEN.seed)
    for _ in range(args.warmup):
        time_oracle_sample(d, steps, pairs_wanted=4, budget_s=1.0, seed=99)
    vals, times = [], []
    desc = cores = None
    for i in range(args.steps):
        v, cores, desc, dt = time_oracle_sample(d, steps, pairs_wanted=64,
                                                budget_s=args.ref_budget, seed=i)
        vals.append(v)
        times.append(dt)
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, same recipe as the GPU arm)",
        "config": {"workload": "varlen: 64 seqs, lengths U[128,8192], H=16, d_k=128, d_v=256, "
                               "+32 decode steps (bounded sample per step)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        barrier()


# ---------------------------------------------------------------- GPU arm
def run_ours(args):
    from gated_delta_rule_45_gb300 import kda
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    init_dist("nccl")
    dev = torch.device("cuda", local)
    kda.load()

    spec, d, steps = make_workload(synth.VARLEN.seed + rank)
    T = int(d["cu_seqlens"][-1])
    N, H, d_k, d_v = spec.num_seqs, spec.H, spec.d_k, spec.d_v
    n_dec = len(steps)
    stream = torch.cuda.Stream(device=dev)

    # device-resident inputs and outputs
    g = {key: d[key].to(dev) for key in ("q", "k", "v", "alpha", "beta", "S0", "cu_seqlens")}
    dec = [{key: st[key].to(dev) for key in ("q", "k", "v", "alpha", "beta")} for st in steps]
    o = torch.empty((T, H, d_v), dtype=torch.bfloat16, device=dev)
    S = torch.empty((N, H, d_v, d_k), dtype=torch.float32, device=dev)
    o_dec = [torch.empty((N, H, d_v), dtype=torch.bfloat16, device=dev) for _ in range(n_dec)]
    wsp = torch.empty(kda.workspace_size(N, H, d_k, d_v, spec.chunk, T), dtype=torch.uint8,
                      device=dev)
    torch.cuda.synchronize()

    ev_pf = []

    def decode_all():
        for i in range(n_dec):
            x = dec[i]
            kda.decode_step(x["q"], x["k"], x["v"], x["alpha"], x["beta"], S, o_dec[i],
                            stream=stream)

    graph = None   # the 32 decode steps as one CUDA graph, once warmed up

    def step(record=False):
        with torch.cuda.stream(stream):
            if record:
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e2 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
            kda.prefill_into(g["q"], g["k"], g["v"], g["alpha"], g["beta"], g["S0"],
                             g["cu_seqlens"], o, S, wsp, chunk=spec.chunk, stream=stream)
            if record:
                e1.record(stream)
            if graph is not None:
                graph.replay()
            else:
                decode_all()
            if record:
                e2.record(stream)
                ev_pf.append((e0, e1, e2))

    for _ in range(args.warmup):
        step()
    kda.device_status(wsp, stream=stream)
    torch.cuda.synchronize()
    try:   # decode steps are ~44 us each: replaying them as a graph saves their launches
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            decode_all()
        torch.cuda.synchronize()
        graph = gr
        for _ in range(2):
            step()
        torch.cuda.synchronize()
    except Exception as exc:   # capture is an optimisation; launches stay correct without it
        print(f"decode graph capture failed ({exc}); launching the steps directly",
              file=sys.stderr)
        graph = None
        torch.cuda.synchronize()

    clocks = ClockSampler(local)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(args.steps):
        step(record=True)
    t_end.record(stream)
    torch.cuda.synchronize()
    clock_info = clocks.stop()
    barrier()
    elapsed = t_start.elapsed_time(t_end) / 1e3
    pf_ms = [e0.elapsed_time(e1) for e0, e1, _ in ev_pf]
    dec_ms = [e1.elapsed_time(e2) for _, e1, e2 in ev_pf]

    tokens_per_step = T + n_dec * N
    elapsed_max, units = reduce_max_sum(elapsed, float(tokens_per_step * args.steps), dev)
    value = units / elapsed_max

    prefill_bytes, decode_bytes = workload_bytes(spec, T, n_dec)
    hbm_peak, peak_src = peaks()
    pf_avg_s = statistics.mean(pf_ms) / 1e3
    achieved = prefill_bytes / pf_avg_s / 1e9
    dec_step_s = statistics.mean(dec_ms) / 1e3 / n_dec

    # end to end: host buffers, copies inside the timed region
    e2e = run_e2e(args, kda, d, steps, spec, dev, stream)
    # the other workloads' kernels, timed alone after the step (one GPU only)
    components_more = {}
    if ws == 1 and not args.no_components:
        components_more = kernel_components(kda, dev, stream, steps=5, warmup=3)
    traffic, traffic_src = stored_traffic()

    if rank == 0:
        # planner + chunk kernel + fast-decay hand-back kernel + one kernel per decode step
        ours_launches = 3 + n_dec
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * elapsed_max / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16",
            "precision": "bf16 inputs and output; tensor-core products on bf16 operands "
                         "(non-input operands as hi + lo bf16 pairs) with fp32 accumulation; "
                         "fp32 state and CUDA-core arithmetic",
            "data": "synthetic (seeded: torch.Generator seed 0 + rank)",
            "config": {"workload": "varlen: 64 seqs, lengths U[128,8192], H=16, d_k=128, "
                                   "d_v=256, chunk=64, S0~N(0,0.1^2), then 32 decode steps",
                       "prefill_tokens": T, "decode_tokens": n_dec * N,
                       "tokens_per_step": tokens_per_step,
                       "l2": "no flush: inputs exceed L2 (%.1f GB per step)"
                             % ((prefill_bytes + n_dec * decode_bytes) / 1e9)},
            "components": {
                "prefill_ms": statistics.mean(pf_ms),
                "prefill_tokens_per_s": T / pf_avg_s,
                "prefill_token_heads_per_s": T * H / pf_avg_s,
                "decode_step_us": dec_step_s * 1e6,
                "decode_state_updates_per_s": N * H / dec_step_s,
                "decode_hbm_gbs": decode_bytes / dec_step_s / 1e9,
                "decode_hbm_frac": decode_bytes / dec_step_s / 1e9 / hbm_peak,
                "kernels_alone": components_more,
            },
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "traffic": traffic,
                         "traffic_source": traffic_src,
                         "kernel": "kda_prefill (planner + chunk kernel)",
                         "algorithmic_bytes_per_launch": prefill_bytes,
                         "peak_source": peak_src + " (MEASURED_PEAKS.json hbm_gbs)"},
            "clocks": clock_info,
            "gpu_launches": ours_launches * args.steps,
            "decode_cuda_graph": graph is not None,
            "e2e": e2e,
        }
        if not args.no_cpu_baseline:
            every = spec.num_seqs * spec.H
            v, cores, desc, _ = time_oracle_sample(d, steps, pairs_wanted=every,
                                                   budget_s=args.cpu_baseline_budget)
            # the same oracle on one thread, over a quarter of the budget
            v1, _, desc1, _ = time_oracle_sample(d, steps, pairs_wanted=every,
                                                 budget_s=args.cpu_baseline_budget / 4, seed=1,
                                                 threads=1)
            line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                                    "sample": desc,
                                    "single_core": {"value": v1, "unit": UNIT, "cores": 1,
                                                    "sample": desc1}}
        print(json.dumps(line), flush=True)


E2E_GROUPS = 8          # sequence groups streamed through the GPU per end-to-end step


def run_e2e(args, kda, d, steps, spec, dev, stream):
    """Same step through the public API with pinned host buffers; H2D of inputs and
    D2H of outputs inside the timed region.

    The batch is cut into E2E_GROUPS groups of consecutive sequences (about equal
    token counts).  Group g's inputs go up on two alternating copy streams while
    group g-1 is prefilled on the compute stream and group g-2's outputs come
    down on a third stream; the 32 decode steps run on the whole batch once every
    group is prefilled, then the state and the decode outputs come down."""
    keys = ("q", "k", "v", "alpha", "beta")
    host = {key: d[key].pin_memory() for key in keys + ("S0",)}
    host_dec = [{key: st[key].pin_memory() for key in keys} for st in steps]
    cu_host = d["cu_seqlens"].to(torch.int64)
    T = int(cu_host[-1])
    N, H, d_k, d_v = spec.num_seqs, spec.H, spec.d_k, spec.d_v
    # groups of consecutive sequences with about equal token counts
    bounds = [0]
    for gi in range(1, E2E_GROUPS):
        n = int(torch.searchsorted(cu_host, T * gi // E2E_GROUPS))
        bounds.append(min(max(n, bounds[-1] + 1), N - (E2E_GROUPS - gi)))
    bounds.append(N)
    groups = [(bounds[i], bounds[i + 1]) for i in range(E2E_GROUPS) if bounds[i + 1] > bounds[i]]
    cu_g_host = [(cu_host[n0:n1 + 1] - cu_host[n0]).to(torch.int32).pin_memory()
                 for n0, n1 in groups]
    g = {key: torch.empty_like(host[key], device=dev) for key in host}
    cu_g = [torch.empty_like(c, device=dev) for c in cu_g_host]
    gd = [{key: torch.empty_like(x[key], device=dev) for key in x} for x in host_dec]
    o = torch.empty((T, H, d_v), dtype=torch.bfloat16, device=dev)
    S = torch.empty((N, H, d_v, d_k), dtype=torch.float32, device=dev)
    o_dec = torch.empty((len(steps), N, H, d_v), dtype=torch.bfloat16, device=dev)
    wsp = torch.empty(kda.workspace_size(N, H, d_k, d_v, spec.chunk, T), dtype=torch.uint8,
                      device=dev)
    o_h = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    S_h = torch.empty(S.shape, dtype=S.dtype).pin_memory()
    od_h = torch.empty(o_dec.shape, dtype=o_dec.dtype).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in host.values()) + \
        sum(x.numel() * x.element_size() for x in cu_g_host) + \
        sum(x.numel() * x.element_size() for hd in host_dec for x in hd.values())
    d2h = sum(x.numel() * x.element_size() for x in (o_h, S_h, od_h))
    up = [torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)]
    down = torch.cuda.Stream(device=dev)

    def step(start_ev):
        for st in up + [down]:
            st.wait_event(start_ev)
        done_down = []
        for gi, (n0, n1) in enumerate(groups):
            t0, t1 = int(cu_host[n0]), int(cu_host[n1])
            cs = up[gi % 2]
            with torch.cuda.stream(cs):
                for key in keys:
                    g[key][t0:t1].copy_(host[key][t0:t1], non_blocking=True)
                g["S0"][n0:n1].copy_(host["S0"][n0:n1], non_blocking=True)
                cu_g[gi].copy_(cu_g_host[gi], non_blocking=True)
                if gi == len(groups) - 1:
                    for i, hd in enumerate(host_dec):
                        for key in hd:
                            gd[i][key].copy_(hd[key], non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(cs)
            stream.wait_event(ev_in)
            with torch.cuda.stream(stream):
                kda.prefill_into(g["q"][t0:t1], g["k"][t0:t1], g["v"][t0:t1],
                                 g["alpha"][t0:t1], g["beta"][t0:t1], g["S0"][n0:n1],
                                 cu_g[gi], o[t0:t1], S[n0:n1], wsp, chunk=spec.chunk,
                                 stream=stream)
                ev_pf = torch.cuda.Event()
                ev_pf.record(stream)
            down.wait_event(ev_pf)
            with torch.cuda.stream(down):
                o_h[t0:t1].copy_(o[t0:t1], non_blocking=True)
        with torch.cuda.stream(stream):
            for i, x in enumerate(gd):
                kda.decode_step(x["q"], x["k"], x["v"], x["alpha"], x["beta"], S, o_dec[i],
                                stream=stream)
            ev_dec = torch.cuda.Event()
            ev_dec.record(stream)
        down.wait_event(ev_dec)
        with torch.cuda.stream(down):
            S_h.copy_(S, non_blocking=True)
            od_h.copy_(o_dec, non_blocking=True)
            ev_end = torch.cuda.Event()
            ev_end.record(down)
        stream.wait_event(ev_end)

    e2e_steps = max(1, min(args.steps, 3))
    ev0 = torch.cuda.Event()
    ev0.record(stream)
    step(ev0)
    torch.cuda.synchronize()
    barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    prev = t0
    for _ in range(e2e_steps):
        step(prev)
        prev = torch.cuda.Event()
        prev.record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    el, units = reduce_max_sum(t0.elapsed_time(t1) / 1e3,
                               float((T + len(steps) * N) * e2e_steps), dev)
    return {"value": units / el, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": e2e_steps,
            "pipeline": f"{len(groups)} sequence groups: H2D on 2 streams, prefill, D2H on a "
                        "third stream, overlapped; decode steps after the last group"}


KERNEL_CASES = ("decode", "prefill", "long", "l2_resident")


def prefill_case(name, kda, dev, stream, gen_device="cpu"):
    """One prefill workload's kernel launch on device-resident inputs: dict(launch,
    nbytes, units, unit, desc, mma_flops, alg_flops).  name: a key of
    synth.WORKLOADS, varlen_prefill, or a gate / update variant of prefill."""
    gate = {"prefill_head_gate": "head", "prefill_log_gate": "log_bf16"}.get(name)
    additive = name == "prefill_additive"
    wname = "varlen" if name == "varlen_prefill" else "prefill" if (gate or additive) else name
    spec = synth.WORKLOADS[wname]
    d = synth.prefill_inputs(spec, device=gen_device)
    g = {key: (d[key].to(dev) if d[key] is not None else None)
         for key in ("q", "k", "v", "alpha", "beta", "S0", "cu_seqlens")}
    del d["q"], d["k"], d["v"], d["alpha"], d["beta"]
    T = int(g["cu_seqlens"][-1])
    o = torch.empty((T, spec.H, spec.d_v), dtype=torch.bfloat16, device=dev)
    S = torch.empty((spec.num_seqs, spec.H, spec.d_v, spec.d_k), device=dev)
    wsp = torch.empty(kda.workspace_size(spec.num_seqs, spec.H, spec.d_k, spec.d_v, spec.chunk,
                                         T), dtype=torch.uint8, device=dev)
    alpha_bytes = None
    if additive:   # the additive update of linear attention on the same inputs
        def launch():
            kda.prefill_additive_into(g["q"], g["k"], g["v"], g["alpha"], g["beta"], g["S0"],
                                      g["cu_seqlens"], o, S, wsp, chunk=spec.chunk,
                                      stream=stream)
    elif gate is None:
        def launch():
            kda.prefill_into(g["q"], g["k"], g["v"], g["alpha"], g["beta"], g["S0"],
                             g["cu_seqlens"], o, S, wsp, chunk=spec.chunk, stream=stream)
    else:
        # the same synthetic gates in the other layout: channel 0's gate for
        # every channel, or log alpha rounded to bf16
        if gate == "head":
            ga = g["alpha"][:, :, 0].contiguous()
            alpha_bytes = 4
        else:
            ga = torch.log(g["alpha"]).to(torch.bfloat16)
            alpha_bytes = spec.d_v * 2

        def launch():
            kda.prefill_gates_into(g["q"], g["k"], g["v"], ga, g["beta"], g["S0"],
                                   g["cu_seqlens"], o, S, wsp, gate=gate, chunk=spec.chunk,
                                   stream=stream)
    nbytes, _ = workload_bytes(spec, T, 0, alpha_bytes)
    desc = (f"{name}: N={spec.num_seqs}, T={T}, H={spec.H}, d_k={spec.d_k}, "
            f"d_v={spec.d_v}, chunk={spec.chunk}"
            + (f", gate layout {gate}" if gate else "")
            + (", additive update (no prediction)" if additive else ""))
    lens = [int(x) for x in d["lengths"]]
    chunks = sum((n + spec.chunk - 1) // spec.chunk for n in lens)
    mma_flops = MMA_FLOPS_PER_BLOCK_CHUNK * spec.H * (spec.d_v // 128) * chunks
    alg_flops = ALG_FLOPS_PER_TOKEN_HEAD * T * spec.H * spec.d_v // 128
    return dict(launch=launch, nbytes=nbytes, units=T, unit="tokens/s", desc=desc,
                mma_flops=mma_flops, alg_flops=alg_flops, token_heads=T * spec.H, d=d,
                inputs=g)


def decode_case(kda, dev, stream, gen_device="cpu"):
    spec = synth.DECODE
    d = synth.decode_inputs(spec, device=gen_device)
    g = {key: d[key].to(dev) for key in ("q", "k", "v", "alpha", "beta", "S")}
    o = torch.empty((spec.B, spec.H, spec.d_v), dtype=torch.bfloat16, device=dev)

    def launch():
        kda.decode_step(g["q"], g["k"], g["v"], g["alpha"], g["beta"], g["S"], o, stream=stream)
    esz = 2
    bh = spec.B * spec.H
    nbytes = bh * (2 * spec.d_k * esz + 2 * spec.d_v * esz + spec.d_v * 4 + 4
                   + 2 * spec.d_v * spec.d_k * 4)
    return dict(launch=launch, nbytes=nbytes, units=bh, unit="state-updates/s",
                desc="decode: B=256, H=32, d_k=d_v=128, bf16, fp32 state in place (1.07 GB)")


def time_launches(launch, stream, steps: int, warmup: int):
    """Mean CUDA-event time (ms) of `launch` on `stream` after `warmup` untimed calls."""
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            launch()
    torch.cuda.synchronize()
    events = []
    with torch.cuda.stream(stream):
        for _ in range(steps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            launch()
            e1.record(stream)
            events.append((e0, e1))
    torch.cuda.synchronize()
    return statistics.mean(e0.elapsed_time(e1) for e0, e1 in events)


def kernel_components(kda, dev, stream, steps: int, warmup: int) -> dict:
    """The other workloads' kernels timed alone (CUDA events), each with its
    throughput and roofline fraction; inputs drawn on the device (same recipe)."""
    hbm_peak, _ = peaks()
    tpeak, _ = bf16_peak()
    out = {}
    for name in KERNEL_CASES:
        c = decode_case(kda, dev, stream, "cuda") if name == "decode" else \
            prefill_case(name, kda, dev, stream, "cuda")
        ms = time_launches(c["launch"], stream, steps, warmup)
        gbs = c["nbytes"] / (ms / 1e3) / 1e9
        r = {"ms": ms, "value": c["units"] / (ms / 1e3), "unit": c["unit"],
             "hbm_gbs": gbs, "hbm_frac": gbs / hbm_peak, "workload": c["desc"]}
        if name != "decode":
            r["token_heads_per_s"] = c["token_heads"] / (ms / 1e3)
        if name == "l2_resident":
            # inputs stay in L2 between launches: the tensor pipe is the roofline;
            # algorithmic flops (dense tiles of the chunk form) and the flops the
            # kernel issues (operand splits included) side by side
            alg = c["alg_flops"] / (ms / 1e3) / 1e12
            iss = c["mma_flops"] / (ms / 1e3) / 1e12
            r.update({"tensor_tflops_algorithmic": alg, "tensor_frac_algorithmic": alg / tpeak,
                      "tensor_tflops_issued": iss, "tensor_frac_issued": iss / tpeak,
                      "tensor_peak_tflops": tpeak})
        out[name] = r
        del c
        torch.cuda.empty_cache()
    return out


def run_component(args):
    """Time one workload's kernel alone (``--workload prefill|long|decode``): the
    other configurations, reported as kernel-level lines next to the full step."""
    from gated_delta_rule_45_gb300 import kda
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    hbm_peak, peak_src = peaks()
    events = []
    if args.workload == "decode":
        c = decode_case(kda, dev, stream)
        launch, nbytes, units, unit, desc = (c["launch"], c["nbytes"], c["units"], c["unit"],
                                             c["desc"])
    elif args.workload in ("attnres", "attnres_small"):
        # Blocked Attention Residuals over a 64-layer network (8 blocks of 8),
        # 16384 tokens of width 2048, bf16; synthetic layer outputs stand in
        # for the layers.  One step = the 64 layers' inputs, called as a model
        # would: block sums stored as they complete, an in-place running sum.
        spec = synth.ATTNRES
        if args.workload == "attnres_small":   # the profiling case: 4096 tokens
            import dataclasses
            spec = dataclasses.replace(spec, T=4096)
        x = synth.attnres_inputs(spec, device=dev)
        T, d = spec.T, spec.d
        nblk = len(spec.block_sizes)
        blocks = torch.empty((nblk + 1, T, d), dtype=torch.bfloat16, device=dev)
        blocks[0] = x["h0"]
        running = torch.empty((T, d), device=dev)
        hbuf = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
        outs, qs = x["outs"], x["queries"]
        calls = []   # (nb, partial, h_last, partial_out, block_out) per layer
        layer = 0
        for n, size in enumerate(spec.block_sizes, start=1):
            for i in range(size):
                if i == 0 and n == 1:
                    calls.append((1, None, None, None, None))
                elif i == 0:
                    calls.append((n - 1, running, outs[layer - 1], None, blocks[n - 1]))
                elif i == 1:
                    calls.append((n, None, outs[layer - 1], running, None))
                else:
                    calls.append((n, running, outs[layer - 1], running, None))
                layer += 1

        def launch():
            for li, (nb, part, last, pout, bout) in enumerate(calls):
                kda.attnres_layer(blocks[:nb], qs[li], partial=part, h_last=last,
                                  partial_out=pout, block_out=bout, h=hbuf, stream=stream)
        row = T * d
        nbytes = 0
        for nb, part, last, pout, bout in calls:
            nbytes += nb * row * 2 + row * 2 + d * 4          # sources, h, q
            nbytes += (row * 4 if part is not None else 0) + (row * 2 if last is not None else 0)
            nbytes += (row * 4 if pout is not None else 0) + (row * 2 if bout is not None else 0)
        units, unit = T, "tokens/s"
        desc = (f"{args.workload}: Blocked Attention Residuals, 64 layers in 8 blocks of 8, T={T}, d={d}, "
                f"bf16 sources and outputs, fp32 running sum; one step = 64 attnres_layer calls")
    elif args.workload in ("backward", "backward_small"):
        spec = synth.PREFILL
        if args.workload == "backward_small":   # the profiling case: 512 tokens per sequence
            import dataclasses
            spec = dataclasses.replace(spec, len_lo=512, len_hi=512)
        d = synth.prefill_inputs(spec)
        dO, dS_T = synth.backward_cotangents(d)
        g = {key: (d[key].to(dev) if d[key] is not None else None)
             for key in ("q", "k", "v", "alpha", "beta", "S0", "cu_seqlens")}
        dO, dS_T = dO.to(dev), dS_T.to(dev)
        T = int(d["cu_seqlens"][-1])
        N, H, d_k, d_v = spec.num_seqs, spec.H, spec.d_k, spec.d_v
        grads = {"dq": torch.empty((T, H, d_k), device=dev),
                 "dk": torch.empty((T, H, d_k), device=dev),
                 "dv": torch.empty((T, H, d_v), device=dev),
                 "dalpha": torch.empty((T, H, d_v), device=dev),
                 "dbeta": torch.empty((T, H), device=dev),
                 "dS0": torch.empty((N, H, d_v, d_k), device=dev)}
        wsp = torch.empty(kda.backward_workspace_size(N, T, H, d_k, d_v, spec.chunk),
                          dtype=torch.uint8, device=dev)

        def launch():
            kda.backward_into(g["q"], g["k"], g["v"], g["alpha"], g["beta"], g["S0"],
                              g["cu_seqlens"], dO, dS_T, grads, wsp, chunk=spec.chunk,
                              stream=stream)
        units, unit = T, "tokens/s"
        nchunks = sum((n + spec.chunk - 1) // spec.chunk for n in d["lengths"])
        # HBM bytes the gradients need at the least: inputs and dO, dS_T read once,
        # the six gradients written once (the workspace traffic is extra)
        state = N * H * d_v * d_k * 4
        nbytes = T * H * (2 * d_k * 2 + 2 * d_v * 2 + d_v * 4 + 4 + 2 * d_k * 4
                          + 2 * d_v * 4 + 4) + 3 * state
        bwd_flops = 2 * BWD_FMA_PER_BLOCK_CHUNK * nchunks * H * (d_v // 64)
        bwd_mma_flops = 2 * BWD_MMA_FMA_PER_BLOCK_CHUNK * nchunks * H * (d_v // 64)
        desc = (f"{args.workload}: kda_backward, N={N}, T={T}, H={H}, d_k={d_k}, d_v={d_v}, "
                f"chunk={spec.chunk}; dO bf16, dS_T fp32; all six gradients fp32")
    else:
        c = prefill_case(args.workload, kda, dev, stream)
        launch, nbytes, units, unit, desc = (c["launch"], c["nbytes"], c["units"], c["unit"],
                                             c["desc"])
        mma_flops, alg_flops = c["mma_flops"], c["alg_flops"]
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            launch()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            launch()
            e1.record(stream)
            events.append((e0, e1))
    torch.cuda.synchronize()
    clock_info = clocks.stop()
    ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in events)
    achieved = nbytes / (ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak, "traffic": None,
                "algorithmic_bytes_per_launch": nbytes, "peak_source": peak_src}
    l2 = "no flush: inputs exceed L2"
    if args.workload in ("backward", "backward_small"):
        # the products run on the tensor cores (bf16 mma.sync): that pipe, not HBM,
        # is the roofline; the algorithmic fp32-equivalent rate is reported beside it
        tpeak, tsrc = bf16_peak()
        tflops = bwd_mma_flops / (ms / 1e3) / 1e12
        roofline = {"bound": "tensor", "achieved": tflops, "peak": tpeak, "unit": "TFLOP/s",
                    "frac": tflops / tpeak, "traffic": None,
                    "mma_flops_per_launch": bwd_mma_flops, "peak_source": tsrc,
                    "algorithmic_flops_per_launch": bwd_flops,
                    "algorithmic_tflops": bwd_flops / (ms / 1e3) / 1e12,
                    "hbm_equivalent_gbs": achieved}
    if args.workload == "l2_resident":
        # inputs stay in L2 between launches: the tensor pipe, not HBM, is the roofline
        tpeak, tsrc = bf16_peak()
        tflops = alg_flops / (ms / 1e3) / 1e12
        roofline = {"bound": "tensor", "achieved": tflops, "peak": tpeak, "unit": "TFLOP/s",
                    "frac": tflops / tpeak, "traffic": None,
                    "algorithmic_flops_per_launch": alg_flops,
                    "issued_mma_flops_per_launch": mma_flops,
                    "issued_tflops": mma_flops / (ms / 1e3) / 1e12,
                    "issued_frac": mma_flops / (ms / 1e3) / 1e12 / tpeak,
                    "peak_source": tsrc, "hbm_equivalent_gbs": achieved}
        l2 = "L2-resident on purpose (~110 MB of inputs and states, relaunched back to back)"
    line = {
        "metric": METRIC, "value": units / (ms / 1e3), "unit": unit, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 in/out; fp32 state", "data": "synthetic (seeded)",
        "config": {"workload": desc, "l2": l2},
        "roofline": roofline,
        "clocks": clock_info, "component_only": True}
    if not args.no_cpu_baseline and args.workload in ("backward", "attnres"):
        # the oracle beside the GPU figure, on a bounded sample of the same workload
        if args.workload == "backward":
            v, cores, cdesc = time_oracle_backward_sample(d, dO.cpu(), dS_T.cpu(),
                                                          args.ref_budget)
        else:
            v, cores, cdesc = time_oracle_attnres_sample(x, calls, args.ref_budget)
        line["cpu_baseline"] = {"value": v, "unit": unit, "cores": cores, "kind": "oracle",
                                "sample": cdesc}
    print(json.dumps(line), flush=True)


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--ref-budget", type=float, default=None,
                   help="seconds of CPU work per reference step / cpu_baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-baseline-budget", type=float, default=15.0,
                   help="seconds of CPU work for the cpu_baseline sample on every core "
                        "(a quarter of it again on one thread)")
    p.add_argument("--no-components", action="store_true",
                   help="skip timing the other workloads' kernels alone after the step")
    p.add_argument("--workload",
                   choices=["varlen", "varlen_prefill", "prefill", "long", "long_small", "decode",
                            "l2_resident", "prefill_head_gate", "prefill_log_gate",
                            "backward", "backward_small", "attnres", "attnres_small",
                            "prefill_additive"],
                   default="varlen",
                   help="varlen (default): the full step; others time one kernel alone "
                        "(varlen_prefill: the varlen batch's prefill without the decode steps; "
                        "l2_resident: the chunk kernel with its inputs in L2, against the "
                        "tensor-core peak; prefill_head_gate / prefill_log_gate: the prefill "
                        "workload with a per-head fp32 gate / a bf16 log-alpha gate; "
                        "long_small: the long workload at 32768 tokens, for profiling the "
                        "sequence-axis split; "
                        "backward: kda_backward on the prefill workload; backward_small: "
                        "the same with 512 tokens per sequence, for profiling; attnres: "
                        "Blocked Attention Residuals over a 64-layer network; attnres_small: "
                        "the same with 4096 tokens, for profiling; prefill_additive: the "
                        "prefill workload under the additive update of linear attention)")
    args = p.parse_args(argv)
    # at least 3 untimed warm-up steps; the JSON line reports the number used
    args.warmup = max(3, args.warmup)
    if args.ref_budget is None:
        args.ref_budget = max(1.0, min(8.0, 120.0 / max(1, args.steps)))
    if args.impl == "reference":
        run_reference(args)
    elif args.workload != "varlen":
        run_component(args)
    else:
        run_ours(args)
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
