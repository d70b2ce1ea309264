"""KDA (Kimi Delta Attention) gated delta-rule recurrence on GB300 (sm_103a).

The computation lives in ``libkda.so`` (CUDA kernels behind the C ABI of ``include/kda.h``);
this package holds its build script, the ctypes binding and the seeded synthetic workloads.
"""
from .binding import (  # noqa: F401
    KdaError,
    Params,
    chunk_prefill,
    check_device_errors,
    commit_verified_states,
    lib,
    make_params,
    prefill_workspace_size,
    recurrent_decode,
    recurrent_verify,
    replay_decode,
    replay_rings,
    selftest_wait_timeout,
    status_string,
)
