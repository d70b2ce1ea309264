"""The replica path of bench.py on two gloo ranks (CPU): rendezvous on 127.0.0.1, the barrier, and
the max-over-ranks reduction that turns per-rank step times into the job's time.  The hot path
has no exchange step, so these helpers are the whole multi-rank logic.  Also the algorithmic byte
counts and the reference arm's line (same metric, unit and config as our arm)."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    r, w, local = bench.dist_env()
    dist = bench.maybe_init_dist(w, "gloo")
    try:
        bench.barrier(dist)
        ms = 1.5 + rank                      # each rank's measured step time
        job_ms = bench.reduce_max(dist, ms, torch.device("cpu"))
        tokens = 1000                        # units each replica processes
        value = w * tokens / (job_ms * 1e-3)
        q.put((r, w, local, job_ms, value))
    finally:
        dist.destroy_process_group()


def test_two_replicas_reduce_to_the_slowest_rank():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for r, (rank, w, local, job_ms, value) in enumerate(res):
        assert (rank, w, local) == (r, world, r)
        assert job_ms == pytest.approx(2.5)          # max over ranks
        assert value == pytest.approx(2 * 1000 / 2.5e-3)


def test_single_process_needs_no_process_group():
    assert bench.maybe_init_dist(1, "gloo") is None
    assert bench.reduce_max(None, 3.0, torch.device("cpu")) == 3.0
    bench.barrier(None)


def test_algorithmic_byte_counts():
    """The per-unit byte counts the roofline uses, against the figures written out by hand."""
    # decode: per (request, head) state read + write, q/k/v bf16, g_raw fp32, b_raw, out bf16
    assert bench.decode_bytes(1, 1, 128, 2, 2) == 2 * 128 * 128 * 4 + 3 * 256 + 512 + 4 + 256 + 4 + 512
    # prefill: 1540 bytes per token and head for bf16 in/out, d = 128, plus the state per sequence
    assert bench.prefill_bytes(1, 0, 1, 128, 2, 2) == 1540 + 4 + 512
    assert bench.prefill_bytes(0, 1, 1, 128, 2, 2) == 2 * 128 * 128 * 4 + 4 + 512
    # verify (per-head gate): one state read, per draft one state write and its token's bytes
    assert bench.verify_bytes(1, 4, 1, 128, 2, 2) == 65536 + 4 * (65536 + 768 + 4 + 4 + 256) + 8


def test_buffered_decode_bytes_follow_the_halving_model():
    """ReplaySSM, section 12: the plain decode reads and writes the whole fp32 state every step; the
    buffered decode reads the checkpoint every step and writes it once per ring of L steps, so with
    staggered cursors its state traffic per step is (1 + 1/L) / 2 of the plain decode's.  The vector
    terms (token inputs, ring entries) fade against it as d grows."""
    for L in (8, 16):
        cursors = list(range(L))                 # one request in L flushes at each step
        for D, tol in ((128, 0.15), (4096, 0.01)):
            ratio = bench.replay_bytes(cursors, L, 1, D, 2, 2) / bench.decode_bytes(L, 1, D, 2, 2)
            assert abs(ratio - (1 + 1 / L) / 2) < tol, (L, D, ratio)


def test_per_kernel_algorithmic_bytes_partition_the_call():
    """The intra kernel's bytes (token inputs once) and the state pass's (states read and written,
    output written) add up to the prefill call's algorithmic bytes: the dominant-kernel roofline
    neither double-counts nor drops a tensor."""
    T, N, H, D = 16412, 8, 32, 128
    for io, out in ((2, 2), (2, 4), (4, 4)):
        call = bench.prefill_bytes(T, N, H, D, io, out)
        assert bench.intra_bytes(T, H, D, io) + bench.state_pass_bytes(T, N, H, D, out) == call
    # per (token, head): q, k, v bf16 + g_raw fp32 + b_raw fp32 = 1284 bytes
    assert bench.intra_bytes(1, 1, 128, 2) - (4 + 128 * 4) == 1284


def test_reference_arm_line_matches_our_arm(monkeypatch, capsys):
    """The reference arm prints one line with our arm's metric, unit, direction and config, so that
    the two lines compare like for like (the oracle's timing is stubbed: no compute here)."""
    import argparse
    import json

    monkeypatch.setattr(bench, "oracle_workload_once", lambda: (0.5, 4, 16412))
    monkeypatch.setattr(bench, "dist_env", lambda: (0, 1, 0))
    import oracle
    monkeypatch.setattr(oracle, "build", lambda *a, **k: None)
    args = argparse.Namespace(gpus=1, steps=3, warmup=1)
    assert bench.run_reference(args) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert (line["metric"], line["unit"], line["higher_is_better"]) == (bench.METRIC, bench.UNIT, True)
    assert line["config"] == bench.headline_config(16412, 1)
    assert line["value"] == pytest.approx(16412 / 0.5)
    assert line["e2e"]["value"] == line["value"] and line["cpu_baseline"]["cores"] == 4
