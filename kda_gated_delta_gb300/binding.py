"""Thin ctypes binding of libkda (include/kda.h).

Argument marshalling only: every step of the computation runs in the CUDA kernels behind the
C ABI.  PyTorch supplies device memory and the current stream.  There is no fallback: if
``libkda.so`` has not been built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

KDA_OK = 0
KDA_F32, KDA_BF16 = 0, 1
GATE_PER_CHANNEL, GATE_PER_HEAD = 0, 1

_STATUS = {
    0: "KDA_OK", -1: "KDA_ERR_INVALID_ARG", -2: "KDA_ERR_UNSUPPORTED", -3: "KDA_ERR_MISALIGNED",
    -4: "KDA_ERR_WORKSPACE", -5: "KDA_ERR_CUDA", -6: "KDA_ERR_DEVICE_CHECK", -7: "KDA_ERR_SCRATCH_LIMIT",
}


class KdaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_STATUS.get(status, status)} ({status_string(status)})")


class Params(ctypes.Structure):
    """Mirror of ``kda_params``."""
    _fields_ = [
        ("num_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("io_dtype", ctypes.c_int32),
        ("out_dtype", ctypes.c_int32),
        ("gate_kind", ctypes.c_int32),
        ("chunk_size", ctypes.c_int32),
        ("use_lower_bound", ctypes.c_int32),
        ("lower_bound", ctypes.c_float),
        ("scale", ctypes.c_float),
        ("l2_eps", ctypes.c_float),
        ("softplus_threshold", ctypes.c_float),
    ]


_P = ctypes.c_void_p
_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Load libkda.so (built by ``kda_gated_delta_gb300.build``); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libkda.so is not built ({path}); run python -m kda_gated_delta_gb300.build")
        L = ctypes.CDLL(path)
        L.kda_params_init.restype = None
        L.kda_params_init.argtypes = [ctypes.POINTER(Params), ctypes.c_int32, ctypes.c_int32]
        L.kda_status_string.restype = ctypes.c_char_p
        L.kda_status_string.argtypes = [ctypes.c_int32]
        L.kda_chunk_prefill_workspace_size.restype = ctypes.c_size_t
        L.kda_chunk_prefill_workspace_size.argtypes = [ctypes.POINTER(Params), ctypes.c_int32, ctypes.c_int64]
        L.kda_chunk_prefill.restype = ctypes.c_int32
        L.kda_chunk_prefill.argtypes = [ctypes.POINTER(Params), _P, _P, _P, _P, _P, _P, _P, _P,
                                        ctypes.c_int32, ctypes.c_int64, _P, ctypes.c_int64, _P, _P,
                                        _P, ctypes.c_size_t, _P]
        L.kda_chunk_prefill_timed.restype = ctypes.c_int32
        L.kda_chunk_prefill_timed.argtypes = L.kda_chunk_prefill.argtypes + [ctypes.POINTER(ctypes.c_void_p)]
        L.kda_recurrent_decode.restype = ctypes.c_int32
        L.kda_recurrent_decode.argtypes = [ctypes.POINTER(Params), _P, _P, _P, _P, _P, _P, _P,
                                           ctypes.c_int32, _P, ctypes.c_int64, _P, _P, _P]
        L.kda_recurrent_verify.restype = ctypes.c_int32
        L.kda_recurrent_verify.argtypes = [ctypes.POINTER(Params), _P, _P, _P, _P, _P, _P, _P,
                                           ctypes.c_int32, ctypes.c_int32, _P, ctypes.c_int64, _P,
                                           _P, _P, _P]
        L.kda_chunk_prefill_snapshots.restype = ctypes.c_int32
        L.kda_chunk_prefill_snapshots.argtypes = L.kda_chunk_prefill.argtypes[:-1] + [_P, ctypes.c_int64, _P]
        L.kda_replay_decode.restype = ctypes.c_int32
        L.kda_replay_decode.argtypes = [ctypes.POINTER(Params), _P, _P, _P, _P, _P, _P, _P, ctypes.c_int32,
                                        _P, ctypes.c_int64, _P, _P, _P, _P, ctypes.c_int32, _P, _P, _P, _P]
        L.kda_commit_verified_states.restype = ctypes.c_int32
        L.kda_commit_verified_states.argtypes = [ctypes.POINTER(Params), _P, ctypes.c_int32, ctypes.c_int32, _P,
                                                 _P, ctypes.c_int64, _P, _P]
        L.kda_check_device_errors.restype = ctypes.c_int32
        L.kda_check_device_errors.argtypes = [_P, ctypes.POINTER(ctypes.c_int32)]
        L.kda_selftest_wait_timeout.restype = ctypes.c_int32
        L.kda_selftest_wait_timeout.argtypes = [ctypes.c_uint32, _P, _P]
        _lib = L
        return L


def status_string(status: int) -> str:
    try:
        return lib().kda_status_string(int(status)).decode()
    except RuntimeError:
        return "library not loaded"


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return KDA_F32
    if dt == torch.bfloat16:
        return KDA_BF16
    raise TypeError(f"unsupported dtype {dt}")


def make_params(num_heads: int, head_dim: int, io_dtype=torch.bfloat16, out_dtype=None,
                gate: str = "kda", chunk_size: int = 64, lower_bound=None, scale=None,
                l2_eps: float = 1e-6, softplus_threshold: float = 20.0) -> Params:
    p = Params()
    lib().kda_params_init(ctypes.byref(p), int(num_heads), int(head_dim))
    p.io_dtype = _dtype_code(io_dtype)
    p.out_dtype = _dtype_code(io_dtype if out_dtype is None else out_dtype)
    p.gate_kind = GATE_PER_CHANNEL if gate == "kda" else GATE_PER_HEAD
    p.chunk_size = int(chunk_size)
    p.use_lower_bound = 0 if lower_bound is None else 1
    p.lower_bound = 0.0 if lower_bound is None else float(lower_bound)
    p.scale = 0.0 if scale is None else float(scale)
    p.l2_eps = float(l2_eps)
    p.softplus_threshold = float(softplus_threshold)
    return p


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _dev(t, name, dtype=None):
    if t is None:
        return
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(rc: int, what: str):
    if rc != KDA_OK:
        raise KdaError(rc, what)


def prefill_workspace_size(params: Params, num_seqs: int, total_tokens: int) -> int:
    return int(lib().kda_chunk_prefill_workspace_size(ctypes.byref(params), int(num_seqs), int(total_tokens)))


PREFILL_PHASE_EVENTS = 4
PREFILL_PHASES = ("chunk_table", "chunk_intra", "chunk_state")


def chunk_prefill(q, k, v, g_raw, b_raw, A_log, dt_bias, cu_seqlens, state_pool, state_idx,
                  out=None, *, params: Params | None = None, workspace=None, stream=None,
                  events=None, chunk_states=None, **kw):
    """kda_chunk_prefill on torch tensors; returns ``out`` ([T, H, D]).  ``state_pool`` is
    updated in place.  ``kw`` are forwarded to :func:`make_params` when ``params`` is None.
    With ``events`` (4 recorded-once ``torch.cuda.Event``), kda_chunk_prefill_timed records them
    around the chunk-table, intra-chunk and state-pass kernels.  With ``chunk_states``
    ([num_chunks, H, D, D] fp32), kda_chunk_prefill_snapshots also writes the state after every
    chunk (chunks numbered by sequence, then position)."""
    T, H, D = q.shape
    if params is None:
        params = make_params(H, D, io_dtype=q.dtype, **kw)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _dev(t, name, q.dtype)
    _dev(g_raw, "g_raw", torch.float32)
    _dev(b_raw, "b_raw", torch.float32)
    _dev(A_log, "A_log", torch.float32)
    _dev(dt_bias, "dt_bias", torch.float32)
    _dev(cu_seqlens, "cu_seqlens", torch.int32)
    _dev(state_pool, "state_pool", torch.float32)
    _dev(state_idx, "state_idx", torch.int32)
    n = state_idx.numel()
    if out is None:
        out = torch.empty((T, H, D), device=q.device,
                          dtype=torch.float32 if params.out_dtype == KDA_F32 else torch.bfloat16)
    _dev(out, "out")
    need = prefill_workspace_size(params, n, T)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _dev(workspace, "workspace", torch.uint8)
    args = (ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(g_raw), _ptr(b_raw), _ptr(A_log),
            _ptr(dt_bias), _ptr(cu_seqlens), n, T, _ptr(state_pool), state_pool.shape[0], _ptr(state_idx),
            _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream))
    if chunk_states is not None:
        if events is not None:
            raise ValueError("events and chunk_states cannot be combined")
        _dev(chunk_states, "chunk_states", torch.float32)
        rc = lib().kda_chunk_prefill_snapshots(*args[:-1], _ptr(chunk_states), chunk_states.shape[0], args[-1])
        _check(rc, "kda_chunk_prefill_snapshots")
        return out
    if events is None:
        rc = lib().kda_chunk_prefill(*args)
    else:
        if len(events) != PREFILL_PHASE_EVENTS:
            raise ValueError("events must hold 4 CUDA events")
        handles = (ctypes.c_void_p * PREFILL_PHASE_EVENTS)(*[ctypes.c_void_p(e.cuda_event) for e in events])
        rc = lib().kda_chunk_prefill_timed(*args, handles)
    _check(rc, "kda_chunk_prefill")
    return out


def recurrent_decode(q, k, v, g_raw, b_raw, A_log, dt_bias, state_pool, state_idx, out=None, *,
                     params: Params | None = None, stream=None, **kw):
    """kda_recurrent_decode: one token per request ([B, H, D] inputs); pool updated in place."""
    B, H, D = q.shape
    if params is None:
        params = make_params(H, D, io_dtype=q.dtype, **kw)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _dev(t, name, q.dtype)
    for name, t in (("g_raw", g_raw), ("b_raw", b_raw), ("A_log", A_log), ("dt_bias", dt_bias),
                    ("state_pool", state_pool)):
        _dev(t, name, torch.float32)
    _dev(state_idx, "state_idx", torch.int32)
    if out is None:
        out = torch.empty((B, H, D), device=q.device,
                          dtype=torch.float32 if params.out_dtype == KDA_F32 else torch.bfloat16)
    _dev(out, "out")
    rc = lib().kda_recurrent_decode(ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(g_raw),
                                    _ptr(b_raw), _ptr(A_log), _ptr(dt_bias), B, _ptr(state_pool),
                                    state_pool.shape[0], _ptr(state_idx), _ptr(out), _stream(stream))
    _check(rc, "kda_recurrent_decode")
    return out


def recurrent_verify(q, k, v, g_raw, b_raw, A_log, dt_bias, state_pool, state_idx, t_draft,
                     inter=None, out=None, *, params: Params | None = None, stream=None, **kw):
    """kda_recurrent_verify: ``t_draft`` tokens per request (request-major rows).  Returns
    ``(out, inter)`` with inter [B, t_draft, H, D, D] fp32; the pool is not modified."""
    TT, H, D = q.shape
    B = state_idx.numel()
    if TT != B * t_draft:
        raise ValueError("q must hold batch * t_draft rows")
    if params is None:
        params = make_params(H, D, io_dtype=q.dtype, **kw)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _dev(t, name, q.dtype)
    for name, t in (("g_raw", g_raw), ("b_raw", b_raw), ("A_log", A_log), ("dt_bias", dt_bias),
                    ("state_pool", state_pool)):
        _dev(t, name, torch.float32)
    _dev(state_idx, "state_idx", torch.int32)
    if inter is None:
        inter = torch.empty((B, t_draft, H, D, D), device=q.device, dtype=torch.float32)
    if out is None:
        out = torch.empty((TT, H, D), device=q.device,
                          dtype=torch.float32 if params.out_dtype == KDA_F32 else torch.bfloat16)
    _dev(inter, "inter", torch.float32)
    _dev(out, "out")
    rc = lib().kda_recurrent_verify(ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(g_raw),
                                    _ptr(b_raw), _ptr(A_log), _ptr(dt_bias), B, int(t_draft),
                                    _ptr(state_pool), state_pool.shape[0], _ptr(state_idx),
                                    _ptr(inter), _ptr(out), _stream(stream))
    _check(rc, "kda_recurrent_verify")
    return out, inter


def replay_rings(num_slots, num_heads, head_dim, ring_len, gate="kda", device="cuda"):
    """Allocate zeroed ReplaySSM rings (d, k, a) for kda_replay_decode."""
    d = torch.zeros(num_slots, num_heads, ring_len, head_dim, device=device)
    k = torch.zeros_like(d)
    a = torch.zeros_like(d) if gate == "kda" else torch.zeros(num_slots, num_heads, ring_len, device=device)
    return d, k, a


def replay_decode(q, k, v, g_raw, b_raw, A_log, dt_bias, state_pool, state_idx, rings, write_pos,
                  force_flush=None, out=None, *, params: Params | None = None, stream=None, **kw):
    """kda_replay_decode: one token per request against checkpoint + ring.  ``rings`` is the
    (ring_d, ring_k, ring_a) triple; ``write_pos`` [B] int32 is not advanced here."""
    B, H, D = q.shape
    ring_d, ring_k, ring_a = rings
    if params is None:
        params = make_params(H, D, io_dtype=q.dtype, **kw)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _dev(t, name, q.dtype)
    for name, t in (("g_raw", g_raw), ("b_raw", b_raw), ("A_log", A_log), ("dt_bias", dt_bias),
                    ("state_pool", state_pool), ("ring_d", ring_d), ("ring_k", ring_k), ("ring_a", ring_a)):
        _dev(t, name, torch.float32)
    _dev(state_idx, "state_idx", torch.int32)
    _dev(write_pos, "write_pos", torch.int32)
    _dev(force_flush, "force_flush", torch.int32)
    if out is None:
        out = torch.empty((B, H, D), device=q.device,
                          dtype=torch.float32 if params.out_dtype == KDA_F32 else torch.bfloat16)
    _dev(out, "out")
    rc = lib().kda_replay_decode(ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(g_raw), _ptr(b_raw),
                                 _ptr(A_log), _ptr(dt_bias), B, _ptr(state_pool), state_pool.shape[0],
                                 _ptr(state_idx), _ptr(ring_d), _ptr(ring_k), _ptr(ring_a), ring_d.shape[2],
                                 _ptr(write_pos), _ptr(force_flush), _ptr(out), _stream(stream))
    _check(rc, "kda_replay_decode")
    return out


def commit_verified_states(inter, accept_len, state_pool, state_idx, *, params: Params | None = None,
                           stream=None, **kw):
    """kda_commit_verified_states: copy inter[b, accept_len[b] - 1] into each accepted slot."""
    B, Td, H, D, _ = inter.shape
    if params is None:
        params = make_params(H, D, **kw)
    _dev(inter, "inter", torch.float32)
    _dev(accept_len, "accept_len", torch.int32)
    _dev(state_pool, "state_pool", torch.float32)
    _dev(state_idx, "state_idx", torch.int32)
    rc = lib().kda_commit_verified_states(ctypes.byref(params), _ptr(inter), B, Td, _ptr(accept_len),
                                          _ptr(state_pool), state_pool.shape[0], _ptr(state_idx), _stream(stream))
    _check(rc, "kda_commit_verified_states")
    return state_pool


def selftest_wait_timeout(polls: int, result=None, stream=None) -> None:
    """Enqueue the bounded-wait self-test (a wait that cannot complete; see kda.h).

    result: None or a device int32 tensor of 2 elements that receives (first wait completed,
    drain completed).  The timeout is then reported by check_device_errors() as code 3."""
    if result is not None:
        _dev(result, "result", torch.int32)
        if result.numel() < 2:
            raise ValueError("result must hold 2 int32 elements")
    rc = lib().kda_selftest_wait_timeout(int(polls), _ptr(result) if result is not None else None,
                                         _stream(stream))
    _check(rc, "kda_selftest_wait_timeout")


def check_device_errors(stream=None) -> int:
    """Synchronise and return the device error code recorded by the kernels (0 = none)."""
    code = ctypes.c_int32(0)
    rc = lib().kda_check_device_errors(_stream(stream), ctypes.byref(code))
    if rc not in (KDA_OK, -6):
        _check(rc, "kda_check_device_errors")
    return int(code.value)
