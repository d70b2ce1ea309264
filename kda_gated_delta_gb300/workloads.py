"""Seeded synthetic inputs for the KDA workloads.

This module only draws random numbers and lays them out; it holds none of the method's
arithmetic (no gate activation, no normalisation, no recurrence).  The same host tensors feed
both the CUDA path and the oracle.

Distributions (the pages' Kimi-Linear shapes, H = 32, d = 128; the tiny case spells them out):
  q, k, v ~ N(0, 1) quantised to the IO dtype;  g_raw ~ N(0, 1) fp32;  b_raw ~ N(0, 1) fp32;
  A_log ~ U(0, ln 16) per head;  dt_bias = 0;  pool slots ~ N(0, 0.01^2) fp32 (std 0.01) or zero;
  state_idx = distinct random slots.  Seeds are 1000 + workload id on a CPU torch.Generator.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass
class Workload:
    wid: int
    name: str
    kind: str                 # "prefill" | "decode" | "verify"
    num_heads: int
    head_dim: int
    io_dtype: torch.dtype
    gate: str = "kda"         # "kda" (per channel) | "gdn" (per head)
    chunk_size: int = 64
    lengths: list = field(default_factory=list)   # prefill: sequence lengths
    batch: int = 0            # decode / verify requests
    t_draft: int = 1          # verify drafts per request
    pool_slots: int = 1
    pool_std: float = 0.0     # 0 -> zeroed slots
    calls: int = 1            # long prefill split into successive calls carrying the state
    description: str = ""


def _lengths_u(gen, n, lo, hi):
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen)]


def workload(wid: int) -> Workload:
    """The five workloads: tiny fp32 prefill, varlen prefill, decode, long chunked prefill,
    scalar-gate verify."""
    gen = torch.Generator().manual_seed(1000 + wid)
    if wid == 0:
        return Workload(0, "tiny_prefill_fp32", "prefill", 2, 16, torch.float32, chunk_size=16,
                        lengths=[64], pool_slots=1, pool_std=0.0,
                        description="1 seq T=64, H=2, d=16, chunk 16, fp32, S0=0")
    if wid == 1:
        return Workload(1, "varlen_prefill_bf16", "prefill", 32, 128, torch.bfloat16, chunk_size=64,
                        lengths=_lengths_u(gen, 8, 512, 4096), pool_slots=512, pool_std=0.01,
                        description="8 seqs, lengths U[512,4096], H=32, d=128, bf16 q/k/v, chunk 64")
    if wid == 2:
        return Workload(2, "decode_bf16", "decode", 32, 128, torch.bfloat16, batch=256,
                        pool_slots=512, pool_std=0.01,
                        description="256 requests x 1 token, H=32, d=128, bf16, 512-slot fp32 pool")
    if wid == 3:
        return Workload(3, "long_chunked_prefill_bf16", "prefill", 32, 128, torch.bfloat16,
                        chunk_size=64, lengths=[131072], calls=32, pool_slots=1, pool_std=0.0,
                        description="1 seq T=131072 as 32 calls x 4096 carrying the state")
    if wid == 4:
        return Workload(4, "gdn_verify_bf16", "verify", 32, 128, torch.bfloat16, gate="gdn",
                        batch=64, t_draft=4, pool_slots=512, pool_std=0.01,
                        description="per-head gate, 64 requests x 4 drafts, intermediate states")
    raise KeyError(wid)


def make_inputs(lengths, num_heads, head_dim, io_dtype, *, gate="kda", pool_slots=1,
                pool_std=0.0, seed=0, dt_bias_std=0.0, padding_rows=(), state_idx=None,
                q_std=1.0, g_mean=0.0, g_std=1.0, b_mean=0.0, b_std=1.0,
                A_log_range=(0.0, math.log(16.0))):
    """Random host inputs for packed sequences of the given lengths.

    ``A_log_range`` = (lo, hi) draws A_log ~ U(lo, hi) (default U(0, ln 16)).
    Returns a dict of CPU tensors: q, k, v [T,H,D] (io_dtype); g_raw [T,H,D] or [T,H]; b_raw [T,H];
    A_log [H]; dt_bias [H,D] or [H]; cu_seqlens [N+1] int32; pool [slots,H,D,D] fp32;
    state_idx [N] int32 (entries listed in ``padding_rows`` set to -1).
    """
    gen = torch.Generator().manual_seed(int(seed))
    T = int(sum(lengths))
    H, D = int(num_heads), int(head_dim)
    N = len(lengths)

    def randn(*shape):
        return torch.randn(*shape, generator=gen, dtype=torch.float32)

    q = (randn(T, H, D) * q_std).to(io_dtype)
    k = (randn(T, H, D) * q_std).to(io_dtype)
    v = randn(T, H, D).to(io_dtype)
    gshape = (T, H, D) if gate == "kda" else (T, H)
    g_raw = randn(*gshape) * g_std + g_mean
    b_raw = randn(T, H) * b_std + b_mean
    lo, hi = float(A_log_range[0]), float(A_log_range[1])
    A_log = torch.rand(H, generator=gen, dtype=torch.float32) * (hi - lo)
    if lo != 0.0:
        A_log = A_log + lo
    dshape = (H, D) if gate == "kda" else (H,)
    dt_bias = randn(*dshape) * dt_bias_std if dt_bias_std > 0 else torch.zeros(dshape, dtype=torch.float32)
    if pool_std > 0:
        pool = randn(pool_slots, H, D, D) * pool_std
    else:
        pool = torch.zeros(pool_slots, H, D, D, dtype=torch.float32)
    if state_idx is None:
        if N > pool_slots:
            raise ValueError("more sequences than pool slots")
        state_idx = torch.randperm(pool_slots, generator=gen)[:N].to(torch.int32)
    else:
        state_idx = torch.as_tensor(state_idx, dtype=torch.int32).clone()
    for r in padding_rows:
        state_idx[r] = -1
    cu = torch.zeros(N + 1, dtype=torch.int32)
    if N:
        cu[1:] = torch.cumsum(torch.as_tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    return dict(q=q, k=k, v=v, g_raw=g_raw, b_raw=b_raw, A_log=A_log, dt_bias=dt_bias,
                cu_seqlens=cu, pool=pool, state_idx=state_idx)


def workload_inputs(wid: int, lengths=None, heads=None):
    """Inputs of workload ``wid`` (optionally with other lengths or head count)."""
    w = workload(wid)
    H = w.num_heads if heads is None else heads
    if w.kind == "prefill":
        lens = w.lengths if lengths is None else lengths
    elif w.kind == "decode":
        lens = [1] * w.batch
    else:
        lens = [w.t_draft] * w.batch
    return make_inputs(lens, H, w.head_dim, w.io_dtype, gate=w.gate, pool_slots=w.pool_slots,
                       pool_std=w.pool_std, seed=1000 + wid)


def to_device(inputs: dict, device) -> dict:
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in inputs.items()}
