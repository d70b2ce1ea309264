"""kda_chunk_prefill_static_scratch: the chunk prefill for callers that cannot allocate device
memory (for example a plugin inside a serving process whose device memory is already handed
out to its own pools).  It uses a fixed scratch array compiled into the library instead of a
caller-provided workspace.

The test calls it through the C ABI, twice in a row on different problems (the second call
finds the first call's leftovers in the shared array), and checks each result against the
ordinary kda_chunk_prefill with a caller-allocated workspace.  Both run the same kernels on the
same inputs, so the outputs and states must be bitwise equal.  It also checks that a problem
larger than the array is rejected before any work is enqueued: the output and the pool keep a
sentinel value and no device error is recorded.  The file is named so that pytest collects it
last."""
import ctypes

import pytest
import torch

from kda_gated_delta_gb300 import binding, build, workloads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
KDA_ERR_SCRATCH_LIMIT = -7
STATIC_SCRATCH_BYTES = 256 << 20


def _lib():
    build.build()
    L = binding.lib()
    f = L.kda_chunk_prefill_static_scratch
    f.restype = ctypes.c_int32
    P = ctypes.c_void_p
    f.argtypes = [ctypes.POINTER(binding.Params), P, P, P, P, P, P, P, P, ctypes.c_int32, ctypes.c_int64,
                  P, ctypes.c_int64, P, P, P]
    return L


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _static_call(L, params, d, pool, out):
    T = d["q"].shape[0]
    n = d["state_idx"].numel()
    return L.kda_chunk_prefill_static_scratch(
        ctypes.byref(params), _ptr(d["q"]), _ptr(d["k"]), _ptr(d["v"]), _ptr(d["g_raw"]), _ptr(d["b_raw"]),
        _ptr(d["A_log"]), _ptr(d["dt_bias"]), _ptr(d["cu_seqlens"]), n, T, _ptr(pool), pool.shape[0],
        _ptr(d["state_idx"]), _ptr(out), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _rel(a, b):
    return ((a.double() - b.double()).abs().max() / b.double().abs().max()).item()


@pytest.mark.parametrize("io", [torch.float32, torch.bfloat16])
def test_static_scratch_matches_workspace_path_twice_in_a_row(io):
    L = _lib()
    H, D = 8, 128
    problems = [
        workloads.make_inputs([700, 33, 129], H, D, io, pool_slots=6, pool_std=0.05, seed=901),
        workloads.make_inputs([64, 5, 1, 200], H, D, io, pool_slots=6, pool_std=0.05, seed=902,
                              padding_rows=(2,)),
    ]
    for inp in problems:                                   # two calls in a row on the shared array
        d = workloads.to_device(inp, DEV)
        T = d["q"].shape[0]
        params = binding.make_params(H, D, io_dtype=io, out_dtype=torch.float32, chunk_size=64)
        assert binding.prefill_workspace_size(params, d["state_idx"].numel(), T) <= STATIC_SCRATCH_BYTES

        pool_s = d["pool"].clone()
        out_s = torch.empty(T, H, D, device=DEV, dtype=torch.float32)
        rc = _static_call(L, params, d, pool_s, out_s)
        assert rc == 0, binding.status_string(rc)

        pool_w = d["pool"].clone()
        out_w = binding.chunk_prefill(d["q"], d["k"], d["v"], d["g_raw"], d["b_raw"], d["A_log"],
                                      d["dt_bias"], d["cu_seqlens"], pool_w, d["state_idx"], params=params)
        torch.cuda.synchronize()
        assert binding.check_device_errors() == 0
        # same kernels, same inputs: anything short of bitwise equality is a scratch-handling bug
        assert torch.equal(out_s, out_w), f"outputs differ (max relative difference {_rel(out_s, out_w):.3e})"
        assert torch.equal(pool_s, pool_w), f"states differ (max relative difference {_rel(pool_s, pool_w):.3e})"


def test_static_scratch_rejects_problems_beyond_its_size():
    L = _lib()
    H, D = 32, 128
    params = binding.make_params(H, D, io_dtype=torch.bfloat16, chunk_size=64)
    T = 8192                                              # needs about 0.31 GB of scratch
    assert binding.prefill_workspace_size(params, 1, T) > STATIC_SCRATCH_BYTES
    q = torch.zeros(T, H, D, dtype=torch.bfloat16, device=DEV)
    g = torch.zeros(T, H, D, dtype=torch.float32, device=DEV)
    b = torch.zeros(T, H, dtype=torch.float32, device=DEV)
    d = dict(q=q, k=q, v=q, g_raw=g, b_raw=b, A_log=torch.zeros(H, device=DEV), dt_bias=None,
             cu_seqlens=torch.tensor([0, T], dtype=torch.int32, device=DEV),
             state_idx=torch.zeros(1, dtype=torch.int32, device=DEV))
    pool = torch.full((1, H, D, D), 3.0, device=DEV)
    out = torch.full((T, H, D), 7.0, dtype=torch.bfloat16, device=DEV)
    binding.check_device_errors()
    assert _static_call(L, params, d, pool, out) == KDA_ERR_SCRATCH_LIMIT
    assert "scratch" in binding.status_string(KDA_ERR_SCRATCH_LIMIT)
    torch.cuda.synchronize()
    # rejected before anything was enqueued: both buffers keep their sentinels, no device error
    assert bool((out == 7.0).all()) and bool((pool == 3.0).all())
    assert binding.check_device_errors() == 0
