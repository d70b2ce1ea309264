#!/usr/bin/env python
"""Benchmark of the KDA hot path on one GB300 (or N replicas under torchrun).

One step = one pass of the whole path over one batch of synthetic input:
  * chunk prefill of the varlen workload (8 sequences, lengths U[512, 4096], H = 32, d = 128,
    bf16 q/k/v, fp32 gates, chunk 64, states from a 512-slot fp32 pool)       -> headline value
  * single-token decode (256 requests, H = 32, d = 128, pool updated in place) -> "decode"
  * scalar-gate verify (64 requests x 4 drafts, intermediate states written)  -> "verify"
  * buffered (ReplaySSM) decode of the decode workload, ring lengths 8 and 16
                                                    -> "decode_replay", "decode_replay_l16"
Every input lives in HBM before the timed region; each working set is larger than the 129 MB
L2, so no L2 flush is needed between steps.  Kernel durations come from CUDA events recorded on
the launching stream (the prefill's three kernels through kda_chunk_prefill_timed).

Outside the timed steps, on rank 0: the tiny fp32 prefill's launch latency ("tiny", us per call)
and the long prefill, 1 sequence of 131072 tokens as 32 successive 4096-token calls carrying
the state ("long_prefill").

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--only prefill|decode]

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 CPU oracle instead, over the
whole varlen workload per step, and prints the same metric.  ``--only prefill`` runs the varlen
prefill alone (no decode, verify, tiny or long workloads, no e2e or CPU baseline) and ``--only
decode`` the decode, verify and buffered-decode kernels alone: small processes for profiler
captures, whose JSON line is not the bench line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefill tokens/s and decode tokens/s (state GB/s, % HBM/tensor roofline)"
UNIT = "tokens/s"


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum, one ncu capture of a bench
# step, caches flushed before each kernel), valid only for the kernel source they were taken on:
# the hash covers the kernel's file and the two headers every kernel file includes.
MEASURED_TRAFFIC = {
    "kda_prefill.cu": {"sha256_16": "fa729363c4e70a4f",
                       "kda_chunk_table": 0.02e6, "kda_chunk_intra": 1257.3e6, "kda_chunk_state": 766.4e6},
    "kda_recurrent.cu": {"sha256_16": "b92d5644c888e5ec",
                         "kda_recurrent_decode": 1022.3e6, "kda_recurrent_verify": 616.9e6,
                         "kda_replay_decode_l8": 643.0e6, "kda_replay_decode_l16": 674.0e6},
}
TRAFFIC_HEADERS = ("kda_internal.cuh", "kda_tc.cuh")


def source_hash(src):
    """First 16 hex digits of the sha256 of a kernel file followed by the shared headers."""
    import hashlib
    h = hashlib.sha256()
    for name in (src,) + TRAFFIC_HEADERS:
        with open(os.path.join(ROOT, "kda_gated_delta_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel):
    """Bytes per launch from the stored capture, or None if the kernel's source changed since."""
    for src, rec in MEASURED_TRAFFIC.items():
        if kernel in rec:
            try:
                h = source_hash(src)
            except OSError:
                return None
            return rec[kernel] if h == rec["sha256_16"] else None
    return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), float(m["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# ---------------------------------------------------------------------------------------------
# algorithmic bytes (mandatory traffic: inputs once, outputs once, each state read + written once)
# ---------------------------------------------------------------------------------------------
def prefill_bytes(T, N_active, H, D, io_bytes, out_bytes):
    per_token_head = 3 * D * io_bytes + D * 4 + 4 + D * out_bytes      # q,k,v + g_raw + b_raw + out
    state = 2 * D * D * 4                                               # read + write per (seq, head)
    params = H * 4 + H * D * 4                                          # A_log, dt_bias
    return T * H * per_token_head + N_active * H * state + params


def intra_bytes(T, H, D, io_bytes):
    """The intra-chunk kernel alone: the prefill's token inputs read once (q, k, v in the IO type,
    g_raw and b_raw fp32) and the gate parameters.  The record it writes for the state pass is
    workspace: it counts against efficiency (traffic), not as algorithmic work."""
    return T * H * (3 * D * io_bytes + D * 4 + 4) + H * 4 + H * D * 4


def state_pass_bytes(T, N_active, H, D, out_bytes):
    """The state pass alone: each (sequence, head) state read and written once, the output written
    once.  The record it reads is workspace."""
    return N_active * H * 2 * D * D * 4 + T * H * D * out_bytes


def decode_bytes(B, H, D, io_bytes, out_bytes):
    return B * H * (2 * D * D * 4 + 3 * D * io_bytes + D * 4 + 4 + D * out_bytes) + H * 4 + H * D * 4


def replay_bytes(write_pos, ring_len, H, D, io_bytes, out_bytes):
    """Bytes of one buffered-decode step: checkpoint read, ring entries read (d, k, a), then either
    the ring append (non-flush) or the checkpoint write (flush), plus the token's inputs/output."""
    total = 0
    for wp in write_pos:
        per = D * D * 4 + wp * 3 * D * 4 + 3 * D * io_bytes + D * 4 + 4 + D * out_bytes
        per += D * D * 4 if wp == ring_len - 1 else 3 * D * 4
        total += H * per
    return total + H * 4 + H * D * 4


def verify_bytes(B, Td, H, D, io_bytes, out_bytes, per_head_gate=True):
    g = 4 if per_head_gate else D * 4
    per_token = D * D * 4 + 3 * D * io_bytes + g + 4 + D * out_bytes    # inter-state write + inputs + out
    return B * H * (D * D * 4 + Td * per_token) + H * 8


# ---------------------------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu = gpu_id
        self.proc = None
        self.file = None

    def start(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu)], stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        self.file.flush()
        self.file.seek(0)
        rows = [l.strip().split(", ") for l in self.file.read().splitlines() if l.strip()]
        self.file.close()
        os.unlink(self.file.name)
        sm, smax, reasons, power = [], [], set(), []
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            if len(r) < 10:
                continue
            try:
                sm.append(float(r[2]))
                smax.append(float(r[3]))
                power.append(float(r[4]))
            except ValueError:
                continue
            for n, val in zip(names, r[6:10]):
                if val.strip().lower() == "active":
                    reasons.add(n)
        # samples under load: the top half by SM clock / power are the timed region's
        loaded = [s for s, p in zip(sm, power) if p >= statistics.median(power)] if power else sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------------------------
# distributed helpers (replicas; the path has no exchange step)
# ---------------------------------------------------------------------------------------------
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def maybe_init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def reduce_max(dist, x, device):
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ---------------------------------------------------------------------------------------------
# CPU oracle timing (baseline and reference arm)
# ---------------------------------------------------------------------------------------------
_PREFILL_HOST = {}


def headline_config(T, world):
    """The `config` of the headline line, the same for our arm and the reference arm."""
    return {"workload": f"varlen_prefill_bf16: 8 seqs, lengths U[512,4096] (seed 1001), T={T}, H=32, d=128, "
                        "chunk 64",
            "io_dtype": "bf16", "out_dtype": "bf16", "state_dtype": "f32", "tokens_per_step": T,
            "l2": "no flush: every working set > 129 MB L2", "parallelism": f"replicas x{world}"}


def oracle_workload_once():
    """Oracle over the whole varlen workload (8 sequences, all 32 heads, threads over heads)."""
    import oracle
    from kda_gated_delta_gb300 import workloads

    if "inp" not in _PREFILL_HOST:
        _PREFILL_HOST["inp"] = workloads.workload_inputs(1)
    inp = _PREFILL_HOST["inp"]
    threads = min(len(os.sched_getaffinity(0)), 32)
    p = oracle.make_params(32, 128)
    t0 = time.perf_counter()
    oracle.forward(p, inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["b_raw"], inp["A_log"], inp["dt_bias"],
                   inp["cu_seqlens"], inp["pool"], inp["state_idx"], nthreads=threads)
    return time.perf_counter() - t0, threads, int(inp["cu_seqlens"][-1])


def cpu_baseline(target_s=10.0):
    """Time the oracle as it stands on a bounded sample: the whole varlen workload, repeated until
    about target_s seconds of CPU time have been spent."""
    total, reps, thr, T = 0.0, 0, 1, 0
    while total < target_s and reps < 64:
        t, thr, T = oracle_workload_once()
        total += t
        reps += 1
    return {"value": T * reps / total, "unit": UNIT, "cores": thr, "kind": "oracle",
            "sample": f"fp64 token recurrence over the whole varlen workload ({T} tokens, 8 sequences, "
                      f"32 heads, threads over heads) x {reps}, {total:.1f} s"}


def run_reference(args):
    """The reference arm of this build: the fp64 oracle (the pages carry no runnable reference),
    timed as it stands on the host cores over the same varlen workload as our arm's headline,
    one whole workload per step."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    for _ in range(args.warmup):
        oracle_workload_once()
    times, thr, T = [], 1, 0
    for _ in range(args.steps):
        t, thr, T = oracle_workload_once()
        times.append(t)
    total = sum(times)
    value = T * args.steps / total
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": headline_config(T, world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": thr, "kind": "oracle",
                             "sample": f"fp64 token recurrence over the whole varlen workload ({T} tokens, "
                                       f"8 sequences, 32 heads, threads over heads) per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------------------------
def _tiny_latency(kda, workloads, dev, reps=200):
    """The tiny fp32 prefill (1 sequence of 64 tokens, H = 2, d = 16, chunk 16): a launch-latency
    figure, in microseconds per call, on the device (events around back-to-back calls) and on the
    host (wall clock per call including the synchronisation at the end)."""
    import torch
    w = workloads.workload(0)
    inp = workloads.to_device(workloads.workload_inputs(0), dev)
    p = kda.make_params(w.num_heads, w.head_dim, io_dtype=torch.float32, out_dtype=torch.float32,
                        chunk_size=w.chunk_size)
    T = int(inp["cu_seqlens"][-1])
    ws = torch.empty(kda.prefill_workspace_size(p, 1, T), dtype=torch.uint8, device=dev)
    out = torch.empty(T, w.num_heads, w.head_dim, dtype=torch.float32, device=dev)
    pool = inp["pool"].clone()

    def call():
        kda.chunk_prefill(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["b_raw"], inp["A_log"], inp["dt_bias"],
                          inp["cu_seqlens"], pool, inp["state_idx"], out, params=p, workspace=ws)

    for _ in range(20):
        call()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    a.record()
    for _ in range(reps):
        call()
    b.record()
    torch.cuda.synchronize()
    host_us = 1e6 * (time.perf_counter() - t0) / reps
    dev_us = 1e3 * a.elapsed_time(b) / reps
    return {"us_per_call": round(dev_us, 2), "host_us_per_call": round(host_us, 2), "launches_per_call": 3,
            "calls": reps, "workload": "tiny_prefill_fp32: 1 seq T=64, H=2, d=16, chunk 16, fp32 in/out",
            "bound": "launch latency (no roofline)"}


def _long_prefill(kda, workloads, dev, roof, reps=2):
    """The long prefill: 1 sequence of 131072 tokens as 32 successive 4096-token calls carrying
    the state in one slot (bf16 in and out, chunk 64).  One untimed pass, then ``reps`` timed
    passes; every call is timed with events on the launching stream."""
    import torch
    w = workloads.workload(3)
    H, D, per = w.num_heads, w.head_dim, 4096
    host = workloads.workload_inputs(3)
    d = workloads.to_device(host, dev)
    del host
    p = kda.make_params(H, D, io_dtype=torch.bfloat16, out_dtype=torch.bfloat16, chunk_size=64)
    ws = torch.empty(kda.prefill_workspace_size(p, 1, per), dtype=torch.uint8, device=dev)
    out = torch.empty(per * w.calls, H, D, dtype=torch.bfloat16, device=dev)
    cu = torch.tensor([0, per], dtype=torch.int32, device=dev)
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(w.calls)] for _ in range(reps + 1)]
    for e in [x for r in evs for c in r for x in c]:
        e.record()
    torch.cuda.synchronize()
    for r in range(reps + 1):
        pool = d["pool"].clone()
        for c in range(w.calls):
            s = slice(c * per, (c + 1) * per)
            kda.chunk_prefill(d["q"][s], d["k"][s], d["v"][s], d["g_raw"][s], d["b_raw"][s], d["A_log"],
                              d["dt_bias"], cu, pool, d["state_idx"], out[s], params=p, workspace=ws, events=evs[r][c])
    torch.cuda.synchronize()
    call_ms, phase = [], [0.0, 0.0, 0.0]
    for r in range(1, reps + 1):
        for c in range(w.calls):
            e = evs[r][c]
            call_ms.append(e[0].elapsed_time(e[3]))
            for j in range(3):
                phase[j] += e[j].elapsed_time(e[j + 1])
    n = len(call_ms)
    ms_call = sum(call_ms) / n
    per_call_B = prefill_bytes(per, 1, H, D, 2, 2)
    rf = roof(per_call_B, ms_call, ("kda_chunk_table", "kda_chunk_intra", "kda_chunk_state"))
    rf["traffic"] = None                       # the stored capture is of the varlen workload
    rf["scope"] = "one 4096-token call: its token inputs and output, the carried state read and written once"
    return {"value": round(per * w.calls / (ms_call * 1e-3 * w.calls), 1), "unit": UNIT,
            "ms_per_call": round(ms_call, 5), "ms_per_call_median": round(statistics.median(call_ms), 5),
            "ms_total": round(ms_call * w.calls, 4), "calls": w.calls, "tokens_per_call": per,
            "phase_ms_per_call": {"kda_chunk_table": round(phase[0] / n, 5), "kda_chunk_intra": round(phase[1] / n, 5),
                                  "kda_chunk_state": round(phase[2] / n, 5)},
            "roofline": rf,
            "workload": "long_chunked_prefill_bf16: 1 seq T=131072 as 32 calls x 4096 carrying the state, "
                        "H=32, d=128, chunk 64, bf16 in/out"}


def run_ours(args):
    import torch

    rank, world, local = dist_env()
    dist = maybe_init_dist(world, "nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from kda_gated_delta_gb300 import build as kbuild
    kbuild.build()
    import kda_gated_delta_gb300 as kda
    from kda_gated_delta_gb300 import workloads

    bw_peak, _, peak_src = peaks()
    H, D = 32, 128
    only_prefill = args.only == "prefill"

    # ---- inputs, resident in HBM --------------------------------------------------------------
    wp, wd, wv = workloads.workload(1), workloads.workload(2), workloads.workload(4)
    pre_h = workloads.workload_inputs(1)
    pre = workloads.to_device(pre_h, dev)
    T = int(pre_h["cu_seqlens"][-1])
    Np = len(wp.lengths)
    p_pre = kda.make_params(H, D, io_dtype=torch.bfloat16, out_dtype=torch.bfloat16, chunk_size=64)
    ws = torch.empty(kda.prefill_workspace_size(p_pre, Np, T), dtype=torch.uint8, device=dev)
    out_pre = torch.empty(T, H, D, dtype=torch.bfloat16, device=dev)
    RLS = (8, 16)
    if not only_prefill:
        dec = workloads.to_device(workloads.workload_inputs(2), dev)
        ver = workloads.to_device(workloads.workload_inputs(4), dev)
        p_dec = kda.make_params(H, D, io_dtype=torch.bfloat16, out_dtype=torch.bfloat16)
        p_ver = kda.make_params(H, D, io_dtype=torch.bfloat16, out_dtype=torch.bfloat16, gate="gdn")
        out_dec = torch.empty(wd.batch, H, D, dtype=torch.bfloat16, device=dev)
        out_ver = torch.empty(wv.batch * wv.t_draft, H, D, dtype=torch.bfloat16, device=dev)
        inter = torch.empty(wv.batch, wv.t_draft, H, D, D, dtype=torch.float32, device=dev)
        # buffered (ReplaySSM) decode on the decode workload at ring lengths 8 (the pages'
        # microbenchmark) and 16 (the pages' default); cursors staggered across requests so that
        # 1/L of the rows flush per step
        rep = {}
        for RL in RLS:
            rpool = dec["pool"].clone()
            rep[RL] = dict(pool=rpool, rings=kda.replay_rings(rpool.shape[0], H, D, RL, device=dev),
                           pos=[torch.tensor([(t + b) % RL for b in range(wd.batch)], dtype=torch.int32, device=dev)
                                for t in range(RL)],
                           out=torch.empty(wd.batch, H, D, dtype=torch.bfloat16, device=dev))

    K, W = args.steps, args.warmup
    ev = lambda: torch.cuda.Event(enable_timing=True)
    pre_ev = [[ev() for _ in range(4)] for _ in range(K + W)]
    dec_ev = [[ev(), ev()] for _ in range(K + W)]
    ver_ev = [[ev(), ev()] for _ in range(K + W)]
    rep_ev = {RL: [[ev(), ev()] for _ in range(K + W)] for RL in RLS}
    for e in [x for row in pre_ev for x in row]:
        e.record()          # create the underlying CUDA events before handing them to the library
    torch.cuda.synchronize()
    launches_per_step = 3 if only_prefill else 3 + 1 + 1 + len(RLS)

    def step(i):
        kda.chunk_prefill(pre["q"], pre["k"], pre["v"], pre["g_raw"], pre["b_raw"], pre["A_log"],
                          pre["dt_bias"], pre["cu_seqlens"], pre["pool"], pre["state_idx"], out_pre,
                          params=p_pre, workspace=ws, events=pre_ev[i])
        if only_prefill:
            return
        dec_ev[i][0].record()
        kda.recurrent_decode(dec["q"], dec["k"], dec["v"], dec["g_raw"], dec["b_raw"], dec["A_log"],
                             dec["dt_bias"], dec["pool"], dec["state_idx"], out_dec, params=p_dec)
        dec_ev[i][1].record()
        ver_ev[i][0].record()
        kda.recurrent_verify(ver["q"], ver["k"], ver["v"], ver["g_raw"], ver["b_raw"], ver["A_log"],
                             ver["dt_bias"], ver["pool"], ver["state_idx"], wv.t_draft, inter, out_ver,
                             params=p_ver)
        ver_ev[i][1].record()
        for RL in RLS:
            r = rep[RL]
            rep_ev[RL][i][0].record()
            kda.replay_decode(dec["q"], dec["k"], dec["v"], dec["g_raw"], dec["b_raw"], dec["A_log"],
                              dec["dt_bias"], r["pool"], dec["state_idx"], r["rings"], r["pos"][i % RL], None,
                              r["out"], params=p_dec)
            rep_ev[RL][i][1].record()

    for i in range(W):
        step(K + i)
    torch.cuda.synchronize()
    if kda.check_device_errors() != 0:
        raise RuntimeError("device error recorded during warm-up")

    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local)
    clocks = ClockSampler(gpu_id)
    clocks.start()
    time.sleep(0.3)
    barrier(dist)
    torch.cuda.synchronize()
    t_start, t_end = ev(), ev()
    t_start.record()
    for i in range(K):
        step(i)
    t_end.record()
    torch.cuda.synchronize()
    barrier(dist)
    clk = clocks.stop()

    def roof(bytes_, ms, kernels_):
        ach = bytes_ / (ms * 1e-3) / 1e9
        tr = [measured_traffic(k) for k in kernels_]
        return {"bound": "hbm", "achieved": round(ach, 1), "peak": bw_peak, "unit": "GB/s",
                "frac": round(ach / bw_peak, 4), "peak_source": f"hbm_gbs ({peak_src})",
                "algorithmic_bytes": bytes_,
                "traffic": None if any(t is None for t in tr) else sum(tr)}

    step_ms = reduce_max(dist, t_start.elapsed_time(t_end) / K, dev)
    ph = [[pre_ev[i][j].elapsed_time(pre_ev[i][j + 1]) for j in range(3)] for i in range(K)]
    phase_ms = [sum(r[j] for r in ph) / K for j in range(3)]
    pre_ms = reduce_max(dist, sum(phase_ms), dev)
    phase_max = [reduce_max(dist, m, dev) for m in phase_ms]
    pre_B = prefill_bytes(T, Np, H, D, 2, 2)
    value = world * T / (pre_ms * 1e-3)

    kernels = [{"name": n, "ms": round(m, 5)} for n, m in
               zip(("kda_chunk_table", "kda_chunk_intra", "kda_chunk_state"), phase_ms)]
    per_kernel = {
        "kda_chunk_intra": (intra_bytes(T, H, D, 2), phase_max[1],
                            "token inputs read once (q, k, v bf16; g_raw, b_raw fp32); its record is workspace"),
        "kda_chunk_state": (state_pass_bytes(T, Np, H, D, 2), phase_max[2],
                            "states read and written once, output written once; the record it reads is workspace"),
    }
    extra = {}
    if not only_prefill:
        dec_ms = reduce_max(dist, sum(dec_ev[i][0].elapsed_time(dec_ev[i][1]) for i in range(K)) / K, dev)
        ver_ms = reduce_max(dist, sum(ver_ev[i][0].elapsed_time(ver_ev[i][1]) for i in range(K)) / K, dev)
        rep_ms = {RL: reduce_max(dist, sum(rep_ev[RL][i][0].elapsed_time(rep_ev[RL][i][1]) for i in range(K)) / K, dev)
                  for RL in RLS}
        dec_B = decode_bytes(wd.batch, H, D, 2, 2)
        ver_B = verify_bytes(wv.batch, wv.t_draft, H, D, 2, 2)
        rep_B = {RL: sum(replay_bytes(rep[RL]["pos"][i % RL].tolist(), RL, H, D, 2, 2) for i in range(K)) / K
                 for RL in RLS}
        kernels += [{"name": "kda_recurrent_decode", "ms": round(dec_ms, 5)},
                    {"name": "kda_recurrent_verify", "ms": round(ver_ms, 5)}]
        kernels += [{"name": f"kda_replay_decode_l{RL}", "ms": round(rep_ms[RL], 5)} for RL in RLS]
        per_kernel["kda_recurrent_decode"] = (dec_B, dec_ms, "decode workload bytes")
        per_kernel["kda_recurrent_verify"] = (ver_B, ver_ms, "verify workload bytes")
        for RL in RLS:
            per_kernel[f"kda_replay_decode_l{RL}"] = (rep_B[RL], rep_ms[RL],
                                                      "buffered decode bytes (averaged over the timed steps)")
        extra["decode"] = {"value": round(world * wd.batch / (dec_ms * 1e-3), 1), "unit": UNIT, "ms": round(dec_ms, 5),
                           "state_gbs": round(wd.batch * H * 2 * D * D * 4 / (dec_ms * 1e-3) / 1e9, 1),
                           "roofline": roof(dec_B, dec_ms, ("kda_recurrent_decode",)),
                           "workload": "decode_bf16: 256 requests x 1 token, H=32, d=128, 512-slot fp32 pool"}
        extra["verify"] = {"value": round(world * wv.batch * wv.t_draft / (ver_ms * 1e-3), 1), "unit": UNIT,
                           "ms": round(ver_ms, 5), "roofline": roof(ver_B, ver_ms, ("kda_recurrent_verify",)),
                           "workload": "gdn_verify_bf16: 64 requests x 4 drafts, per-head gate, inter states"}
        for RL in RLS:
            key = "decode_replay" if RL == 8 else f"decode_replay_l{RL}"
            extra[key] = {"value": round(world * wd.batch / (rep_ms[RL] * 1e-3), 1), "unit": UNIT,
                          "ms": round(rep_ms[RL], 5), "ring_len": RL,
                          "speedup_vs_decode": round(dec_ms / rep_ms[RL], 3),
                          "roofline": roof(rep_B[RL], rep_ms[RL], (f"kda_replay_decode_l{RL}",)),
                          "workload": f"decode_bf16 through the buffered decode: ring {RL}, cursors staggered, "
                                      f"1/{RL} of the rows flush per step (averaged over the timed steps)"}
    tot = sum(k["ms"] for k in kernels)
    for k in kernels:
        k["share"] = round(k["ms"] / tot, 4)
    dominant = max(kernels, key=lambda k: k["ms"])

    call_roof = roof(pre_B, pre_ms, ("kda_chunk_table", "kda_chunk_intra", "kda_chunk_state"))
    call_roof.update({"scope": "prefill call (chunk_table + chunk_intra + chunk_state), varlen workload",
                      "ms": round(pre_ms, 5)})
    # the dominant kernel's own roofline: its algorithmic bytes over its own event-timed duration
    if dominant["name"] in per_kernel:
        b_, ms_, what = per_kernel[dominant["name"]]
        roofline = roof(b_, ms_, (dominant["name"],))
        roofline.update({"scope": f"dominant kernel {dominant['name']}: {what}", "ms": round(ms_, 5),
                         "dominant_kernel": dominant["name"], "prefill_call": call_roof})
    else:
        roofline = dict(call_roof, dominant_kernel=dominant["name"])

    # ---- end to end: host buffers, copies inside the timed region -----------------------------
    # Every step copies its own inputs host -> device and its output device -> host (pinned host
    # buffers).  Consecutive steps are pipelined on three streams with two device buffer sets: the
    # inputs of step i + 1 travel while step i computes and the output of step i - 1 travels back.
    e2e = None
    if not args.no_e2e and not only_prefill:
        names = ("q", "k", "v", "g_raw", "b_raw", "cu_seqlens", "state_idx")
        host = {k: pre_h[k].pin_memory() for k in names}
        host_out = torch.empty(T, H, D, dtype=torch.bfloat16).pin_memory()
        dbuf = [{k: torch.empty_like(pre[k]) for k in names} for _ in range(2)]
        dout = [torch.empty_like(out_pre) for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = host_out.numel() * host_out.element_size()
        comp = torch.cuda.current_stream()
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]

        def e2e_run(n, start_event=None):
            def issue_in(j):
                with torch.cuda.stream(s_in):
                    if j >= 2:
                        s_in.wait_event(ev_comp[j & 1])       # step j - 2 is done with this buffer set
                    for k_ in names:
                        dbuf[j & 1][k_].copy_(host[k_], non_blocking=True)
                    ev_in[j & 1].record(s_in)

            if start_event is not None:
                s_in.wait_event(start_event)
            issue_in(0)
            for i in range(n):
                b_ = i & 1
                if i + 1 < n:
                    issue_in(i + 1)
                comp.wait_event(ev_in[b_])
                if i >= 2:
                    comp.wait_event(ev_out[b_])               # output of step i - 2 has left dout[b_]
                d_ = dbuf[b_]
                kda.chunk_prefill(d_["q"], d_["k"], d_["v"], d_["g_raw"], d_["b_raw"], pre["A_log"],
                                  pre["dt_bias"], d_["cu_seqlens"], pre["pool"], d_["state_idx"], dout[b_],
                                  params=p_pre, workspace=ws)
                ev_comp[b_].record(comp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_comp[b_])
                    host_out.copy_(dout[b_], non_blocking=True)
                    ev_out[b_].record(s_out)
            comp.wait_stream(s_in)
            comp.wait_stream(s_out)

        e2e_run(W)
        torch.cuda.synchronize()
        barrier(dist)
        a, b = ev(), ev()
        a.record()
        e2e_run(K, start_event=a)
        b.record()
        torch.cuda.synchronize()
        e2e_ms = reduce_max(dist, a.elapsed_time(b) / K, dev)
        e2e = {"value": world * T / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
               "scope": "kda_chunk_prefill through the C ABI with pinned host inputs/outputs; every step "
                        "copies its inputs in and its output out, consecutive steps pipelined on 3 streams"}

    if rank != 0:
        return 0
    if not only_prefill:
        # single-GPU figures outside the timed steps: launch latency and the long chunked prefill
        del dec, ver, inter, rep
        torch.cuda.empty_cache()
        extra["tiny"] = _tiny_latency(kda, workloads, dev)
        extra["long_prefill"] = _long_prefill(kda, workloads, dev, roof)
        if kda.check_device_errors() != 0:
            raise RuntimeError("device error recorded in the tiny or long prefill")
    cpu = None
    if not args.no_cpu_baseline and world == 1 and not only_prefill:
        cpu = cpu_baseline()

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(step_ms, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": headline_config(T, world),
        "roofline": roofline,
        **extra,
        "kernels": kernels,
        "clocks": clk,
        "e2e": e2e,
        "gpu_launches": launches_per_step * K,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_decode_only(args):
    """--only decode: the decode, verify and buffered-decode kernels on their workloads, without the
    prefill workload, so that a profiler capture of them holds a few GB instead of eight.  Prints one
    JSON line with each kernel's time and roofline fraction (a profiling aid, not the bench line)."""
    import torch

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    from kda_gated_delta_gb300 import build as kbuild
    kbuild.build()
    import kda_gated_delta_gb300 as kda
    from kda_gated_delta_gb300 import workloads

    bw_peak, _, _ = peaks()
    H, D = 32, 128
    wd, wv = workloads.workload(2), workloads.workload(4)
    dec = workloads.to_device(workloads.workload_inputs(2), dev)
    ver = workloads.to_device(workloads.workload_inputs(4), dev)
    p_dec = kda.make_params(H, D, io_dtype=torch.bfloat16, out_dtype=torch.bfloat16)
    p_ver = kda.make_params(H, D, io_dtype=torch.bfloat16, out_dtype=torch.bfloat16, gate="gdn")
    out_dec = torch.empty(wd.batch, H, D, dtype=torch.bfloat16, device=dev)
    out_ver = torch.empty(wv.batch * wv.t_draft, H, D, dtype=torch.bfloat16, device=dev)
    inter = torch.empty(wv.batch, wv.t_draft, H, D, D, dtype=torch.float32, device=dev)
    RL = 8
    rpool = dec["pool"].clone()
    rings = kda.replay_rings(rpool.shape[0], H, D, RL, device=dev)
    pos = [torch.tensor([(t + b) % RL for b in range(wd.batch)], dtype=torch.int32, device=dev) for t in range(RL)]
    out_rep = torch.empty(wd.batch, H, D, dtype=torch.bfloat16, device=dev)
    K, W = args.steps, args.warmup
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K + W)]

    def step(i):
        ev[i][0].record()
        kda.recurrent_decode(dec["q"], dec["k"], dec["v"], dec["g_raw"], dec["b_raw"], dec["A_log"],
                             dec["dt_bias"], dec["pool"], dec["state_idx"], out_dec, params=p_dec)
        ev[i][1].record()
        kda.recurrent_verify(ver["q"], ver["k"], ver["v"], ver["g_raw"], ver["b_raw"], ver["A_log"],
                             ver["dt_bias"], ver["pool"], ver["state_idx"], wv.t_draft, inter, out_ver, params=p_ver)
        ev[i][2].record()
        kda.replay_decode(dec["q"], dec["k"], dec["v"], dec["g_raw"], dec["b_raw"], dec["A_log"],
                          dec["dt_bias"], rpool, dec["state_idx"], rings, pos[i % RL], None, out_rep, params=p_dec)
        ev[i][3].record()

    for i in range(W):
        step(K + i)
    torch.cuda.synchronize()
    for i in range(K):
        step(i)
    torch.cuda.synchronize()
    if kda.check_device_errors() != 0:
        raise RuntimeError("device error recorded")
    ms = [sum(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(K)) / K for j in range(3)]
    byts = (decode_bytes(wd.batch, H, D, 2, 2), verify_bytes(wv.batch, wv.t_draft, H, D, 2, 2),
            sum(replay_bytes(pos[i % RL].tolist(), RL, H, D, 2, 2) for i in range(K)) / K)
    line = {"mode": "decode only (profiling aid)", "steps": K, "warmup": W,
            "kernels": [{"name": n, "ms": round(m, 5), "hbm_frac": round(b / (m * 1e-3) / 1e9 / bw_peak, 4)}
                        for n, m, b in zip(("kda_recurrent_decode", "kda_recurrent_verify", "kda_replay_decode_l8"),
                                           ms, byts)]}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default="all", choices=["all", "prefill", "decode"],
                    help="prefill: the varlen prefill alone; decode: decode, verify and buffered decode alone "
                         "(both for profiler captures)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.only == "decode":
        return run_decode_only(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
