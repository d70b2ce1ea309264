"""GPU parity at addresses beyond 32 bits, through the C ABI.

* State slots whose tile starts past 2^31 floats (8 GiB) of an 8.6 GB pool: prefill (tensor-core
  pair), decode, verify, buffered decode and the commit of verified states read and write those
  slots and no other.
* One prefill call of 70,038 tokens over 32 heads, whose per-(chunk, head) workspace records run
  past 2^31 bytes.

The oracle runs on a small pool (the used slots renumbered 0..n-1) and, for the long call, on a
subset of heads sliced out of the inputs; heads are independent in the recurrence, so both are
exact restatements of the same computation."""
import pytest
import torch

import kda_gated_delta_gb300 as kda
from kda_gated_delta_gb300 import workloads
import oracle
from helpers import NTHREADS, PER_HEAD_BF16, np64, oracle_run, per_head_err, rel_err, tol_for

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
H, D = 32, 128
NUM_SLOTS = 4100                                   # slot 4099 starts at 4099 * 32 * 128 * 128 floats
BIG = [4099, 0, 4098, 2050]


def _big_pool(small_pool):
    """The small host pool's slots placed at BIG in a zeroed NUM_SLOTS-slot device pool."""
    assert (max(BIG) * H * D * D) > 2 ** 31
    pool = torch.zeros(NUM_SLOTS, H, D, D, device=DEV, dtype=torch.float32)
    pool[torch.tensor(BIG, device=DEV)] = small_pool.to(DEV)
    return pool


def _others_untouched(pool):
    """Every slot outside BIG still zero (checked on the device)."""
    per_slot = pool.abs().amax(dim=(1, 2, 3))
    per_slot[torch.tensor(BIG, device=DEV)] = 0.0
    return bool((per_slot == 0).all())


def _inputs(lengths, seed, **kw):
    return workloads.make_inputs(lengths, H, D, torch.bfloat16, pool_slots=len(BIG), pool_std=0.05,
                                 seed=seed, dt_bias_std=0.5, state_idx=list(range(len(BIG))), **kw)


def _call_args(d):
    return (d["q"], d["k"], d["v"], d["g_raw"], d["b_raw"], d["A_log"], d["dt_bias"])


def test_state_slots_beyond_2_31_floats():
    big_idx = torch.tensor(BIG, dtype=torch.int32, device=DEV)
    tol = tol_for(torch.bfloat16, torch.float32)

    # prefill: ragged lengths around the chunk size
    inp = _inputs([100, 65, 1, 130], seed=71)
    d = workloads.to_device(inp, DEV)
    pool = _big_pool(inp["pool"])
    out = kda.chunk_prefill(*_call_args(d), d["cu_seqlens"], pool, big_idx, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert kda.check_device_errors() == 0
    o_ref, p_ref, _ = oracle_run(inp, H, D)
    assert rel_err(np64(out), o_ref) <= tol
    assert rel_err(np64(pool[big_idx.long()]), p_ref) <= tol
    assert per_head_err(np64(pool[big_idx.long()]), p_ref) <= PER_HEAD_BF16
    assert _others_untouched(pool)

    # decode: one token per request, from fresh host states in the same slots
    inp = _inputs([1, 1, 1, 1], seed=72)
    d = workloads.to_device(inp, DEV)
    pool = _big_pool(inp["pool"])
    out = kda.recurrent_decode(*_call_args(d), pool, big_idx, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert kda.check_device_errors() == 0
    o_dec, p_dec, _ = oracle_run(inp, H, D)
    assert rel_err(np64(out), o_dec) <= tol
    assert rel_err(np64(pool[big_idx.long()]), p_dec) <= tol
    assert _others_untouched(pool)

    # buffered decode at ring length 8 on the same inputs: an appending step leaves the checkpoint
    # as it was; a forced flush with an empty ring writes the decoded state
    pool = _big_pool(inp["pool"])
    before = pool[big_idx.long()].clone()
    rings = kda.replay_rings(NUM_SLOTS, H, D, 8, device=DEV)
    wp = torch.zeros(len(BIG), dtype=torch.int32, device=DEV)
    out = kda.replay_decode(*_call_args(d), pool, big_idx, rings, wp, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert kda.check_device_errors() == 0
    assert rel_err(np64(out), o_dec) <= tol
    assert torch.equal(pool[big_idx.long()], before) and _others_untouched(pool)
    flush = torch.ones(len(BIG), dtype=torch.int32, device=DEV)
    out = kda.replay_decode(*_call_args(d), pool, big_idx, rings, wp, force_flush=flush, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert kda.check_device_errors() == 0
    assert rel_err(np64(out), o_dec) <= tol
    assert rel_err(np64(pool[big_idx.long()]), p_dec) <= tol
    assert _others_untouched(pool)

    # verify (4 drafts per request; the pool is read, not written) and the commit of accepted states
    Td = 4
    inp = _inputs([Td] * len(BIG), seed=73)
    d = workloads.to_device(inp, DEV)
    pool = _big_pool(inp["pool"])
    before = pool[big_idx.long()].clone()
    out, inter = kda.recurrent_verify(*_call_args(d), pool, big_idx, Td, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert kda.check_device_errors() == 0
    o_ver, _, i_ref = oracle_run(inp, H, D, inter=True)
    assert rel_err(np64(out), o_ver) <= tol
    assert rel_err(np64(inter).reshape(len(BIG) * Td, H, D, D), i_ref) <= tol
    assert torch.equal(pool[big_idx.long()], before) and _others_untouched(pool)
    accept = torch.tensor([1, 4, 2, 3], dtype=torch.int32, device=DEV)
    kda.commit_verified_states(inter, accept, pool, big_idx)
    torch.cuda.synchronize()
    assert kda.check_device_errors() == 0
    for b, acc in enumerate(accept.tolist()):
        assert torch.equal(pool[BIG[b]], inter[b, acc - 1])
    assert _others_untouched(pool)


def test_long_call_workspace_beyond_2_31_bytes():
    lengths = [70001, 37]                          # 1094 + 1 chunks of 64; a ragged tail of 49
    T = sum(lengths)
    params = kda.make_params(H, D)
    assert kda.prefill_workspace_size(params, len(lengths), T) > 2 ** 31
    inp = workloads.make_inputs(lengths, H, D, torch.bfloat16, pool_slots=2, pool_std=0.05, seed=74,
                                dt_bias_std=0.5)
    d = workloads.to_device(inp, DEV)
    pool = d["pool"].clone()
    out = kda.chunk_prefill(*_call_args(d), d["cu_seqlens"], pool, d["state_idx"], out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert kda.check_device_errors() == 0
    # the oracle on three heads sliced out of the inputs (the last one holds the highest records)
    hs = [0, 17, 31]
    sub = dict(inp)
    for n in ("q", "k", "v", "g_raw"):
        sub[n] = inp[n][:, hs].contiguous()
    sub["b_raw"] = inp["b_raw"][:, hs].contiguous()
    sub["A_log"] = inp["A_log"][hs].contiguous()
    sub["dt_bias"] = inp["dt_bias"][hs].contiguous()
    sub["pool"] = inp["pool"][:, hs].contiguous()
    p = oracle.make_params(len(hs), D)
    o_ref, p_ref, _ = oracle.forward(p, sub["q"], sub["k"], sub["v"], sub["g_raw"], sub["b_raw"], sub["A_log"],
                                     sub["dt_bias"], sub["cu_seqlens"], sub["pool"], sub["state_idx"],
                                     nthreads=NTHREADS)
    got_o = np64(out[:, hs])
    got_s = np64(pool[:, hs])
    tol = tol_for(torch.bfloat16, torch.float32)
    assert rel_err(got_o, o_ref) <= tol
    assert rel_err(got_s, p_ref) <= tol
    e_oh = per_head_err(got_o, o_ref, inp["cu_seqlens"].tolist())
    e_sh = per_head_err(got_s, p_ref)
    print(f"70,038-token call, heads {hs}: per-head output {e_oh:.3e}, state {e_sh:.3e}")
    assert e_oh <= PER_HEAD_BF16 and e_sh <= PER_HEAD_BF16, (e_oh, e_sh)
