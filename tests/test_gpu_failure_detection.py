"""Failure detection on the GPU without a fault: a bounded wait that cannot complete gives up,
the kernel records device error 3 (timeout), drains, frees its TMEM and returns; the host reads
the code through kda_check_device_errors, and the context stays usable (a tensor-core prefill
that allocates TMEM on every SM still matches the oracle afterwards)."""
import pytest
import torch

import kda_gated_delta_gb300 as kda
from kda_gated_delta_gb300 import workloads
from helpers import np64, oracle_run, rel_err, tol_for

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("polls", [1, 64, 4096])
def test_bounded_wait_gives_up_and_is_reported(polls):
    kda.check_device_errors()                                        # start from a clear word
    res = torch.full((2,), -1, dtype=torch.int32, device=DEV)
    kda.selftest_wait_timeout(polls, res)
    assert kda.check_device_errors() == 3                            # timeout, read by the host
    assert res.tolist() == [0, 1]                                    # wait gave up; drain completed
    assert kda.check_device_errors() == 0                            # the read cleared it


def test_context_usable_after_timeout():
    kda.check_device_errors()
    for _ in range(4):                                               # TMEM freed on every exit
        kda.selftest_wait_timeout(16)
    assert kda.check_device_errors() == 3
    H, D = 4, 128
    inp = workloads.make_inputs([150, 64, 9], H, D, torch.bfloat16, pool_slots=5, pool_std=0.05, seed=77,
                                dt_bias_std=0.5)
    d = workloads.to_device(inp, DEV)
    pool = d["pool"].clone()
    out = kda.chunk_prefill(d["q"], d["k"], d["v"], d["g_raw"], d["b_raw"], d["A_log"], d["dt_bias"],
                            d["cu_seqlens"], pool, d["state_idx"], chunk_size=64, out_dtype=torch.float32)
    assert kda.check_device_errors() == 0
    o_ref, p_ref, _ = oracle_run(inp, H, D)
    assert rel_err(np64(out), o_ref) <= tol_for(torch.bfloat16, torch.float32)
    assert rel_err(np64(pool), p_ref) <= tol_for(torch.bfloat16, torch.float32)


def test_selftest_argument_checks():
    with pytest.raises(kda.KdaError):
        kda.selftest_wait_timeout(0)
    with pytest.raises(kda.KdaError):
        kda.selftest_wait_timeout((1 << 24) + 1)
    with pytest.raises(ValueError):
        kda.selftest_wait_timeout(8, torch.zeros(1, dtype=torch.int32, device=DEV))
