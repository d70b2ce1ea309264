"""GPU parity of the two prefix-cache / speculative-decoding helpers against the fp64 oracle:

* kda_chunk_prefill_snapshots: the state after every chunk equals the oracle's state after the
  chunk's last token (the oracle's per-token state buffer);
* kda_commit_verified_states after kda_recurrent_verify: each accepted slot equals the oracle
  run over the request's accepted prefix only; accept_len = 0 leaves the slot untouched."""
import numpy as np
import pytest
import torch

import kda_gated_delta_gb300 as kda
from kda_gated_delta_gb300 import workloads
from helpers import np64, oracle_run, rel_err, tol_for

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("io,C,D", [(torch.bfloat16, 64, 128), (torch.float32, 64, 128), (torch.float32, 16, 32)])
def test_chunk_boundary_snapshots(io, C, D):
    H = 3
    lengths = [130, 64, 1, 77]
    inp = workloads.make_inputs(lengths, H, D, io, pool_slots=6, pool_std=0.05, seed=71, dt_bias_std=0.3)
    nchunks = sum((l + C - 1) // C for l in lengths)
    d = workloads.to_device(inp, DEV)
    pool = d["pool"].clone()
    snaps = torch.full((nchunks, H, D, D), float("nan"), device=DEV)
    out = kda.chunk_prefill(d["q"], d["k"], d["v"], d["g_raw"], d["b_raw"], d["A_log"], d["dt_bias"],
                            d["cu_seqlens"], pool, d["state_idx"], chunk_size=C, out_dtype=torch.float32,
                            chunk_states=snaps)
    torch.cuda.synchronize()
    assert kda.check_device_errors() == 0
    o_ref, p_ref, _ = oracle_run(inp, H, D)
    _, _, inter_ref = oracle_run(inp, H, D, inter=True)       # per-token states (pool untouched)
    tol = tol_for(io, torch.float32)
    assert rel_err(np64(out), o_ref) <= tol
    assert rel_err(np64(pool), p_ref) <= tol
    cu = inp["cu_seqlens"].tolist()
    rows, c = [], 0
    for i, L in enumerate(lengths):
        for m in range((L + C - 1) // C):
            rows.append(cu[i] + min((m + 1) * C, L) - 1)
            c += 1
    assert c == nchunks
    assert rel_err(np64(snaps), inter_ref[rows]) <= tol


def test_snapshot_table_too_small_is_recorded():
    H, D = 2, 128
    inp = workloads.make_inputs([200], H, D, torch.bfloat16, pool_slots=1, seed=72)
    d = workloads.to_device(inp, DEV)
    snaps = torch.zeros((2, H, D, D), device=DEV)                   # needs 4 entries
    kda.check_device_errors()
    kda.chunk_prefill(d["q"], d["k"], d["v"], d["g_raw"], d["b_raw"], d["A_log"], d["dt_bias"],
                      d["cu_seqlens"], d["pool"].clone(), d["state_idx"], chunk_size=64, chunk_states=snaps)
    assert kda.check_device_errors() == 2


@pytest.mark.parametrize("gate", ["kda", "gdn"])
def test_commit_accepted_prefix(gate):
    H, D, B, Td = 4, 128, 9, 4
    inp = workloads.make_inputs([Td] * B, H, D, torch.bfloat16, gate=gate, pool_slots=12, pool_std=0.05,
                                seed=73, dt_bias_std=0.3, padding_rows=(7,))
    accept = torch.tensor([0, 1, 2, 3, 4, 4, 1, 2, 3], dtype=torch.int32)
    d = workloads.to_device(inp, DEV)
    pool = d["pool"].clone()
    _, inter = kda.recurrent_verify(d["q"], d["k"], d["v"], d["g_raw"], d["b_raw"], d["A_log"], d["dt_bias"],
                                    pool, d["state_idx"], Td, gate=gate, out_dtype=torch.float32)
    kda.commit_verified_states(inter, accept.to(DEV), pool, d["state_idx"], gate=gate)
    torch.cuda.synchronize()
    assert kda.check_device_errors() == 0
    # oracle: each request run over its accepted prefix only
    sel = [b * Td + t for b in range(B) for t in range(int(accept[b]))]
    sub = dict(inp)
    for n in ("q", "k", "v", "g_raw", "b_raw"):
        sub[n] = inp[n][sel]
    cu = torch.zeros(B + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(accept, 0)
    sub["cu_seqlens"] = cu
    _, p_ref, _ = oracle_run(sub, H, D, gate=gate)
    got = np64(pool)
    changed = [int(inp["state_idx"][b]) for b in range(B) if int(accept[b]) > 0 and b != 7]
    assert rel_err(got[changed], p_ref[changed]) <= tol_for(torch.bfloat16, torch.float32)
    untouched = [s for s in range(12) if s not in changed]
    assert np.array_equal(got[untouched], inp["pool"].double().numpy()[untouched])


def test_commit_rejects_bad_accept_len():
    H, D, B, Td = 2, 64, 3, 2
    inter = torch.randn(B, Td, H, D, D, device=DEV)
    pool = torch.zeros(4, H, D, D, device=DEV)
    sidx = torch.tensor([0, 1, 2], dtype=torch.int32, device=DEV)
    kda.check_device_errors()
    kda.commit_verified_states(inter, torch.tensor([1, 3, -1], dtype=torch.int32, device=DEV), pool, sidx)
    assert kda.check_device_errors() == 4
    assert torch.equal(pool[0], inter[0, 0]) and torch.all(pool[1:] == 0)
