"""GPU parity of kda_recurrent_decode and kda_recurrent_verify against the fp64 oracle, through the
C ABI, on the same seeded host inputs; plus the mode invariances the pages state (verify equals
step-by-step decode, the pool is not modified by verify)."""
import numpy as np
import pytest
import torch

import kda_gated_delta_gb300 as kda
from kda_gated_delta_gb300 import workloads
import math

from helpers import PER_HEAD_BF16, np64, oracle_run, per_head_err, rel_err, tol_for

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def run_decode(inp, gate="kda", out_dtype=torch.float32, lower_bound=None):
    d = workloads.to_device(inp, DEV)
    pool = d["pool"].clone()
    out = kda.recurrent_decode(d["q"], d["k"], d["v"], d["g_raw"], d["b_raw"], d["A_log"], d["dt_bias"],
                               pool, d["state_idx"], gate=gate, out_dtype=out_dtype, lower_bound=lower_bound)
    torch.cuda.synchronize()
    return out, pool


@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("io", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("gate", ["kda", "gdn"])
def test_decode_small(D, io, gate):
    H, B = 3, 7
    inp = workloads.make_inputs([1] * B, H, D, io, gate=gate, pool_slots=11, pool_std=0.3, seed=100 + D,
                                dt_bias_std=0.5, padding_rows=(2,))
    out, pool = run_decode(inp, gate=gate)
    o_ref, p_ref, _ = oracle_run(inp, H, D, gate=gate)
    tol = tol_for(io, torch.float32)
    assert rel_err(np64(out), o_ref) <= tol
    assert rel_err(np64(pool), p_ref) <= tol
    assert np.all(np64(out)[2] == 0.0)                              # padding row
    slots = set(inp["state_idx"].tolist())
    for s in range(11):                                             # untouched slots bit-identical
        if s not in slots or s == -1:
            assert torch.equal(pool[s].cpu(), inp["pool"][s])


def test_decode_bf16_output_and_safe_gate():
    H, D, B = 4, 128, 9
    inp = workloads.make_inputs([1] * B, H, D, torch.bfloat16, pool_slots=16, pool_std=0.5, seed=5,
                                dt_bias_std=2.0)
    out, pool = run_decode(inp, out_dtype=torch.bfloat16, lower_bound=-5.0)
    o_ref, p_ref, _ = oracle_run(inp, H, D, lower_bound=-5.0)
    assert out.dtype == torch.bfloat16
    assert rel_err(np64(out), o_ref) <= tol_for(torch.bfloat16, torch.bfloat16)
    assert rel_err(np64(pool), p_ref) <= tol_for(torch.bfloat16, torch.float32)


def test_decode_full_workload():
    """256 requests x 1 token, H = 32, d = 128, bf16, 512-slot pool: the bench's decode launch."""
    inp = workloads.workload_inputs(2)
    out, pool = run_decode(inp, out_dtype=torch.bfloat16)
    o_ref, p_ref, _ = oracle_run(inp, 32, 128)
    assert rel_err(np64(out), o_ref) <= tol_for(torch.bfloat16, torch.bfloat16)
    assert rel_err(np64(pool), p_ref) <= tol_for(torch.bfloat16, torch.float32)
    out32, pool32 = run_decode(inp, out_dtype=torch.float32)
    assert rel_err(np64(out32), o_ref) <= tol_for(torch.bfloat16, torch.float32)
    # per (request, head), each normalised by its own largest reference value
    used = inp["state_idx"].long()
    e_oh = per_head_err(np64(out32), o_ref, inp["cu_seqlens"].tolist())
    e_sh = per_head_err(np64(pool32)[used], p_ref[used])
    print(f"decode per-head worst: output {e_oh:.3e}, state {e_sh:.3e}")
    assert e_oh <= PER_HEAD_BF16 and e_sh <= PER_HEAD_BF16, (e_oh, e_sh)


@pytest.mark.parametrize("gate,io", [("kda", torch.bfloat16), ("kda", torch.float32), ("gdn", torch.bfloat16)])
def test_decode_softplus_threshold(gate, io):
    """g_raw + dt_bias mostly above the softplus threshold of 20 (some below), with small rates
    (A_log ~ U(ln 0.005, ln 0.05)) so that the decays stay moderate."""
    H, D, B = 4, 128, 12
    inp = workloads.make_inputs([1] * B, H, D, io, gate=gate, pool_slots=16, pool_std=0.3, seed=21,
                                g_mean=21.0, g_std=3.0, dt_bias_std=1.0,
                                A_log_range=(math.log(0.005), math.log(0.05)))
    x = inp["g_raw"] + (inp["dt_bias"][None] if gate == "kda" else inp["dt_bias"][None, :])
    assert (x > 20).float().mean() > 0.5 and (x <= 20).any()
    out, pool = run_decode(inp, gate=gate)
    o_ref, p_ref, _ = oracle_run(inp, H, D, gate=gate)
    tol = tol_for(io, torch.float32)
    assert rel_err(np64(out), o_ref) <= tol
    assert rel_err(np64(pool), p_ref) <= tol


def test_decode_out_of_range_slot_is_recorded():
    H, D = 2, 32
    inp = workloads.make_inputs([1, 1], H, D, torch.float32, pool_slots=4, pool_std=0.1, seed=8,
                                state_idx=[1, 9])
    kda.check_device_errors()
    out, pool = run_decode(inp)
    assert kda.check_device_errors() == 1
    assert kda.check_device_errors() == 0                           # read clears it
    assert np.all(np64(out)[1] == 0.0)
    assert torch.equal(pool[[0, 2, 3]].cpu(), inp["pool"][[0, 2, 3]])


def run_verify(inp, t_draft, gate, out_dtype=torch.float32):
    d = workloads.to_device(inp, DEV)
    pool = d["pool"].clone()
    out, inter = kda.recurrent_verify(d["q"], d["k"], d["v"], d["g_raw"], d["b_raw"], d["A_log"],
                                      d["dt_bias"], pool, d["state_idx"], t_draft, gate=gate,
                                      out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert torch.equal(pool, d["pool"])                            # the pool is never written
    return out, inter


@pytest.mark.parametrize("gate", ["gdn", "kda"])
@pytest.mark.parametrize("D,io", [(16, torch.float32), (64, torch.bfloat16), (128, torch.float32)])
def test_verify_small(gate, D, io):
    H, B, Td = 2, 5, 3
    inp = workloads.make_inputs([Td] * B, H, D, io, gate=gate, pool_slots=7, pool_std=0.2, seed=31 + D,
                                dt_bias_std=0.3, padding_rows=(4,))
    out, inter = run_verify(inp, Td, gate)
    o_ref, _, i_ref = oracle_run(inp, H, D, gate=gate, inter=True)
    tol = tol_for(io, torch.float32)
    assert rel_err(np64(out), o_ref) <= tol
    inter_np = np64(inter).reshape(B * Td, H, D, D)
    valid = [b for b in range(B) if b != 4]
    rows = [b * Td + t for b in valid for t in range(Td)]
    assert rel_err(inter_np[rows], i_ref[rows]) <= tol
    assert np.all(np64(out)[4 * Td:5 * Td] == 0.0)


@pytest.mark.parametrize("gate", ["kda", "gdn"])
@pytest.mark.parametrize("Td", [1, 16])
def test_verify_draft_count_bounds(gate, Td):
    """t_draft at both ends of its range (1 and 16) at d = 128: outputs and every intermediate state
    against the oracle, then the commit of the last draft's state against the oracle's state after
    that draft."""
    H, D, B = 4, 128, 5
    inp = workloads.make_inputs([Td] * B, H, D, torch.bfloat16, gate=gate, pool_slots=7, pool_std=0.05,
                                seed=91 + Td, dt_bias_std=0.3, padding_rows=(3,))
    out, inter = run_verify(inp, Td, gate)
    assert kda.check_device_errors() == 0
    o_ref, _, i_ref = oracle_run(inp, H, D, gate=gate, inter=True)
    tol = tol_for(torch.bfloat16, torch.float32)
    assert rel_err(np64(out), o_ref) <= tol
    inter_np = np64(inter).reshape(B * Td, H, D, D)
    valid = [b for b in range(B) if b != 3]
    rows = [b * Td + t for b in valid for t in range(Td)]
    assert rel_err(inter_np[rows], i_ref[rows]) <= tol
    assert np.all(np64(out)[3 * Td:4 * Td] == 0.0)
    d = workloads.to_device(inp, DEV)
    pool = d["pool"].clone()
    accept = torch.full((B,), Td, dtype=torch.int32, device=DEV)
    kda.commit_verified_states(inter, accept, pool, d["state_idx"], gate=gate)
    torch.cuda.synchronize()
    assert kda.check_device_errors() == 0
    for b in valid:
        s = int(inp["state_idx"][b])
        assert rel_err(np64(pool[s]), i_ref[b * Td + Td - 1]) <= tol


def test_verify_full_workload_gdn():
    """Scalar-gate verify: 64 requests x 4 drafts, H = 32, d = 128, all intermediate states."""
    inp = workloads.workload_inputs(4)
    out, inter = run_verify(inp, 4, "gdn", out_dtype=torch.bfloat16)
    o_ref, _, i_ref = oracle_run(inp, 32, 128, gate="gdn", inter=True)
    assert rel_err(np64(out), o_ref) <= tol_for(torch.bfloat16, torch.bfloat16)
    inter_np = np64(inter).reshape(256, 32, 128, 128)
    assert rel_err(inter_np, i_ref) <= tol_for(torch.bfloat16, torch.float32)
    e_sh = per_head_err(inter_np, i_ref)                    # per (token, head) intermediate state
    print(f"verify per-head worst intermediate state: {e_sh:.3e}")
    assert e_sh <= PER_HEAD_BF16, e_sh


@pytest.mark.parametrize("gate", ["gdn", "kda"])
def test_verify_equals_sequential_decodes_bitwise(gate):
    """The pages' verify test: target_verify equals step-by-step decode, exactly in fp32."""
    H, D, B, Td = 4, 128, 6, 4
    inp = workloads.make_inputs([Td] * B, H, D, torch.float32, gate=gate, pool_slots=8, pool_std=0.2,
                                seed=77)
    out_v, inter = run_verify(inp, Td, gate)
    d = workloads.to_device(inp, DEV)
    pool = d["pool"].clone()
    for t in range(Td):
        rows = torch.arange(B, device=DEV) * Td + t
        sel = lambda x: x[rows].contiguous()
        o = kda.recurrent_decode(sel(d["q"]), sel(d["k"]), sel(d["v"]), sel(d["g_raw"]), sel(d["b_raw"]),
                                 d["A_log"], d["dt_bias"], pool, d["state_idx"], gate=gate,
                                 out_dtype=torch.float32)
        assert torch.equal(o, out_v[rows])
        for b in range(B):
            assert torch.equal(pool[int(inp["state_idx"][b])], inter[b, t])
