"""Shared test helpers: run the oracle and the CUDA path on the same seeded host inputs and
measure the error the way the tolerances are stated (max |gpu - ref| / max |ref| per tensor)."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle

NTHREADS = max(1, len(os.sched_getaffinity(0)))

# Tolerances: fp32 inputs 1e-5; bf16 inputs with fp32 output 2e-3; a bf16 output adds its own
# rounding, at most one bf16 unit in the last place relative to the largest output (2^-8).
TOL_F32 = 1e-5
TOL_BF16 = 2e-3
TOL_BF16_OUT = 2e-3 + 2.0 ** -8
# Per (sequence, head) error of the bf16-input workloads, each block normalised by its own
# largest reference value (a stricter reading than the tensor-wide metric).
PER_HEAD_BF16 = 2e-3


def rel_err(gpu, ref) -> float:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), "non-finite values in the GPU result"
    denom = np.abs(ref).max()
    if denom == 0.0:
        return float(np.abs(gpu).max())
    return float(np.abs(gpu - ref).max() / denom)


def per_head_err(gpu, ref, cu=None) -> float:
    """Worst error over (sequence, head) blocks, each normalised by its own max |ref| (blocks whose
    reference is all zero, i.e. padding, are skipped).  Outputs [T, H, D] are cut into sequences by
    ``cu`` (cu_seqlens); states [S, H, D, D] (``cu`` None) give one block per (slot, head)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), "non-finite values in the GPU result"
    if cu is None:
        n, h = ref.shape[0], ref.shape[1]
        diff = np.abs(gpu - ref).reshape(n, h, -1).max(axis=2)
        den = np.abs(ref).reshape(n, h, -1).max(axis=2)
    else:
        cu = [int(x) for x in cu]
        rows = [(cu[i], cu[i + 1]) for i in range(len(cu) - 1) if cu[i + 1] > cu[i]]
        if not rows:
            return 0.0
        diff = np.stack([np.abs(gpu[a:b] - ref[a:b]).max(axis=(0, 2)) for a, b in rows])
        den = np.stack([np.abs(ref[a:b]).max(axis=(0, 2)) for a, b in rows])
    mask = den > 0
    return float((diff[mask] / den[mask]).max()) if mask.any() else 0.0


def np64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def oracle_run(inp, H, D, gate="kda", lower_bound=None, inter=False, heads=None, scale=0.0):
    p = oracle.make_params(H, D, gate_kind=oracle.GATE_PER_CHANNEL if gate == "kda" else oracle.GATE_PER_HEAD,
                           lower_bound=lower_bound, scale=scale)
    return oracle.forward(p, inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["b_raw"], inp["A_log"],
                          inp["dt_bias"], inp["cu_seqlens"], inp["pool"], inp["state_idx"], inter=inter,
                          heads=heads, nthreads=NTHREADS)


def tol_for(io_dtype, out_dtype):
    if io_dtype == torch.float32:
        return TOL_F32 if out_dtype == torch.float32 else TOL_BF16_OUT
    return TOL_BF16 if out_dtype == torch.float32 else TOL_BF16_OUT
