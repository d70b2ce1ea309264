"""GPU parity of kda_replay_decode (ReplaySSM buffered decode): with ring length 1 it computes
exactly what kda_recurrent_decode computes; with longer rings every step's output equals the
oracle's token-by-token output, and after a final forced flush the checkpoint equals the
oracle's state.  The cursor is advanced on the host by the documented rule."""
import numpy as np
import pytest
import torch

import kda_gated_delta_gb300 as kda
from kda_gated_delta_gb300 import workloads
from helpers import np64, oracle_run, rel_err, tol_for

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _step_rows(inp, B, steps, t):
    rows = torch.arange(B) * steps + t
    return {n: inp[n][rows].contiguous().to(DEV) for n in ("q", "k", "v", "g_raw", "b_raw")}


@pytest.mark.parametrize("gate,D", [("kda", 128), ("gdn", 128), ("kda", 32), ("gdn", 64)])
def test_ring_length_one_is_plain_decode(gate, D):
    H, B, steps = 4, 6, 5
    inp = workloads.make_inputs([steps] * B, H, D, torch.float32, gate=gate, pool_slots=8, pool_std=0.2, seed=81)
    d = workloads.to_device(inp, DEV)
    pool_a, pool_b = d["pool"].clone(), d["pool"].clone()
    rings = kda.replay_rings(8, H, D, 1, gate=gate, device=DEV)
    wp = torch.zeros(B, dtype=torch.int32, device=DEV)
    for t in range(steps):
        x = _step_rows(inp, B, steps, t)
        o1 = kda.recurrent_decode(x["q"], x["k"], x["v"], x["g_raw"], x["b_raw"], d["A_log"], d["dt_bias"],
                                  pool_a, d["state_idx"], gate=gate, out_dtype=torch.float32)
        o2 = kda.replay_decode(x["q"], x["k"], x["v"], x["g_raw"], x["b_raw"], d["A_log"], d["dt_bias"],
                               pool_b, d["state_idx"], rings, wp, gate=gate, out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2)
        assert torch.equal(pool_a, pool_b)


@pytest.mark.parametrize("H", [1, 7])
def test_replay_odd_head_counts(H):
    """d = 128 runs two CTAs per (request, head); with one head and with an odd head count each CTA
    still finds its request, head and half of the rows."""
    D, L, B, steps = 128, 8, 5, 12
    inp = workloads.make_inputs([steps] * B, H, D, torch.bfloat16, pool_slots=6, pool_std=0.05, seed=600 + H,
                                dt_bias_std=0.3)
    o_ref, p_ref, _ = oracle_run(inp, H, D)
    d = workloads.to_device(inp, DEV)
    pool = d["pool"].clone()
    rings = kda.replay_rings(6, H, D, L, device=DEV)
    pos = np.zeros(B, dtype=np.int32)
    tol = tol_for(torch.bfloat16, torch.float32)
    for t in range(steps):
        force = np.zeros(B, dtype=np.int32) if t < steps - 1 else np.ones(B, dtype=np.int32)
        x = _step_rows(inp, B, steps, t)
        o = kda.replay_decode(x["q"], x["k"], x["v"], x["g_raw"], x["b_raw"], d["A_log"], d["dt_bias"], pool,
                              d["state_idx"], rings, torch.tensor(pos, device=DEV), torch.tensor(force, device=DEV),
                              out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert rel_err(np64(o), o_ref[np.arange(B) * steps + t]) <= tol, t
        pos = np.where((pos == L - 1) | (force != 0), 0, pos + 1).astype(np.int32)
    assert kda.check_device_errors() == 0
    used = inp["state_idx"].long()
    assert rel_err(np64(pool)[used], p_ref[used]) <= tol


@pytest.mark.parametrize("gate,io,L,D", [("kda", torch.bfloat16, 8, 128), ("kda", torch.float32, 16, 128),
                                          ("gdn", torch.bfloat16, 4, 128), ("kda", torch.float32, 8, 16),
                                          ("gdn", torch.bfloat16, 8, 32), ("kda", torch.float32, 5, 64),
                                          ("kda", torch.bfloat16, 32, 128)])
def test_replay_matches_oracle_over_many_steps(gate, io, L, D):
    H, B, steps = 4, 7, 21
    inp = workloads.make_inputs([steps] * B, H, D, io, gate=gate, pool_slots=10, pool_std=0.05, seed=82,
                                dt_bias_std=0.3, padding_rows=(5,))
    o_ref, p_ref, _ = oracle_run(inp, H, D, gate=gate)             # token-by-token over each request
    d = workloads.to_device(inp, DEV)
    pool = d["pool"].clone()
    rings = kda.replay_rings(10, H, D, L, gate=gate, device=DEV)
    pos = np.zeros(B, dtype=np.int32)
    tol = tol_for(io, torch.float32)
    rng = np.random.default_rng(5)
    for t in range(steps):
        force = (rng.random(B) < 0.1).astype(np.int32)
        if t == steps - 1:
            force[:] = 1                                            # end with a checkpoint
        x = _step_rows(inp, B, steps, t)
        wp = torch.tensor(pos, device=DEV)
        o = kda.replay_decode(x["q"], x["k"], x["v"], x["g_raw"], x["b_raw"], d["A_log"], d["dt_bias"], pool,
                              d["state_idx"], rings, wp, torch.tensor(force, device=DEV), gate=gate,
                              out_dtype=torch.float32)
        torch.cuda.synchronize()
        ref_t = o_ref[np.arange(B) * steps + t]
        assert rel_err(np64(o), ref_t) <= tol, t
        flushed = (pos == L - 1) | (force != 0)
        pos = np.where(flushed, 0, pos + 1).astype(np.int32)
    assert kda.check_device_errors() == 0
    valid = [int(inp["state_idx"][b]) for b in range(B) if b != 5]
    assert rel_err(np64(pool)[valid], p_ref[valid]) <= tol


def test_replay_bad_write_pos_is_recorded():
    H, D, B = 2, 64, 3
    inp = workloads.make_inputs([1] * B, H, D, torch.float32, pool_slots=4, pool_std=0.1, seed=83)
    d = workloads.to_device(inp, DEV)
    pool = d["pool"].clone()
    rings = kda.replay_rings(4, H, D, 4, device=DEV)
    kda.check_device_errors()
    o = kda.replay_decode(d["q"], d["k"], d["v"], d["g_raw"], d["b_raw"], d["A_log"], d["dt_bias"], pool,
                          d["state_idx"], rings, torch.tensor([0, 4, 1], dtype=torch.int32, device=DEV),
                          out_dtype=torch.float32)
    assert kda.check_device_errors() == 5
    assert torch.all(o[1] == 0)
    assert torch.equal(pool, d["pool"])                              # no row flushed
