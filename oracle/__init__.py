"""fp64 CPU oracle of the KDA gated delta-rule recurrence (ctypes wrapper of kda_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the benchmark's
CPU-baseline leg import this module; the product path never does.  The oracle shares no code
with the CUDA library: it is compiled from ``kda_oracle.c`` with the host C compiler.

Inputs are the same quantised tensors the CUDA path receives (bf16 or fp32), widened exactly
to fp64 here.  The recurrence follows "linear_attention" (zdszero.github.io), sections
"统一递归形式" and "KDA：逐通道的遗忘门"; see ``kda_oracle.c`` for the passage behind each step.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libkda_oracle.so")
# A test can point the wrapper at another build of kda_oracle.c (the mutation test does).
_SO_OVERRIDE = os.environ.get("KDA_ORACLE_LIB")
_lock = threading.Lock()
_lib = None

GATE_PER_CHANNEL = 0
GATE_PER_HEAD = 1


def build(force: bool = False) -> str:
    """Compile kda_oracle.c into a shared library with gcc (portable flags only)."""
    src = os.path.join(_HERE, "kda_oracle.c")
    hdr = os.path.join(_HERE, "kda_oracle.h")
    os.makedirs(_BUILD, exist_ok=True)
    fresh = (os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(src)
             and os.path.getmtime(_SO) >= os.path.getmtime(hdr))
    if fresh and not force:
        return _SO
    tmp = _SO + f".{os.getpid()}.tmp"
    # -ffp-contract=off: no fused multiply-adds, so the fp64 results are the same on x86 and Arm.
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


class Params(ctypes.Structure):
    _fields_ = [
        ("num_heads", ctypes.c_int32),
        ("dk", ctypes.c_int32),
        ("dv", ctypes.c_int32),
        ("gate_kind", ctypes.c_int32),
        ("use_lower_bound", ctypes.c_int32),
        ("use_qk_l2norm", ctypes.c_int32),
        ("lower_bound", ctypes.c_double),
        ("scale", ctypes.c_double),
        ("l2_eps", ctypes.c_double),
        ("softplus_threshold", ctypes.c_double),
    ]


def make_params(num_heads, dk, dv=None, gate_kind=GATE_PER_CHANNEL, lower_bound=None,
                scale=0.0, l2_eps=1e-6, softplus_threshold=20.0, use_qk_l2norm=True) -> Params:
    p = Params()
    p.num_heads = int(num_heads)
    p.dk = int(dk)
    p.dv = int(dk if dv is None else dv)
    p.gate_kind = int(gate_kind)
    p.use_lower_bound = 0 if lower_bound is None else 1
    p.lower_bound = 0.0 if lower_bound is None else float(lower_bound)
    p.use_qk_l2norm = 1 if use_qk_l2norm else 0
    p.scale = float(scale)
    p.l2_eps = float(l2_eps)
    p.softplus_threshold = float(softplus_threshold)
    return p


_D = ctypes.POINTER(ctypes.c_double)
_I = ctypes.POINTER(ctypes.c_int32)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = _SO_OVERRIDE or build()
            L = ctypes.CDLL(path)
            L.kdao_softplus.restype = ctypes.c_double
            L.kdao_softplus.argtypes = [ctypes.c_double, ctypes.c_double]
            L.kdao_sigmoid.restype = ctypes.c_double
            L.kdao_sigmoid.argtypes = [ctypes.c_double]
            L.kdao_gate.restype = None
            L.kdao_gate.argtypes = [ctypes.POINTER(Params), ctypes.c_int, _D, _D, ctypes.c_double, _D]
            L.kdao_l2_normalize.restype = None
            L.kdao_l2_normalize.argtypes = [ctypes.c_int, _D, ctypes.c_double, ctypes.c_double, _D]
            L.kdao_unified_step.restype = None
            L.kdao_unified_step.argtypes = [ctypes.c_int, ctypes.c_int, _D, _D, ctypes.c_double,
                                            ctypes.c_double, _D, _D, _D, _D]
            L.kdao_forward.restype = ctypes.c_int
            L.kdao_forward.argtypes = [ctypes.POINTER(Params), _D, _D, _D, _D, _D, _D, _D, _I,
                                       ctypes.c_int32, _D, ctypes.c_int64, _I, _D, _D,
                                       ctypes.c_int32, ctypes.c_int32]
            L.kdao_chunk_forward.restype = ctypes.c_int
            L.kdao_chunk_forward.argtypes = [ctypes.POINTER(Params), ctypes.c_int32, _D, _D, _D, _D,
                                             _D, _D, _D, _I, ctypes.c_int32, _D, ctypes.c_int64,
                                             _I, _D, ctypes.c_int32, ctypes.c_int32]
            _lib = L
    return _lib


def _f64(a):
    """Contiguous fp64 numpy copy of a numpy array or a CPU torch tensor (exact widening)."""
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().to("cpu")
        import torch  # local: the oracle itself does not need torch
        a = a.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a):
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _dp(a):
    return None if a is None else a.ctypes.data_as(_D)


def _ip(a):
    return a.ctypes.data_as(_I)


def softplus(x, threshold=20.0):
    return lib().kdao_softplus(float(x), float(threshold))


def sigmoid(x):
    return lib().kdao_sigmoid(float(x))


def gate(params: Params, a, dt_bias, A_log_h):
    a = _f64(a).reshape(-1)
    dt = None if dt_bias is None else _f64(dt_bias).reshape(-1)
    g = np.empty_like(a)
    lib().kdao_gate(ctypes.byref(params), a.size, _dp(a), _dp(dt), float(A_log_h), _dp(g))
    return g


def l2_normalize(x, eps=1e-6, scale=1.0):
    x = _f64(x).reshape(-1)
    out = np.empty_like(x)
    lib().kdao_l2_normalize(x.size, _dp(x), float(eps), float(scale), _dp(out))
    return out


def unified_step(S, gamma, alpha_w, beta_w, k, v, q):
    """One unified-recurrence step on a [dk][dv] fp64 state (in place); returns o."""
    assert S.dtype == np.float64 and S.flags.c_contiguous
    dk, dv = S.shape
    gamma = _f64(gamma).reshape(-1)
    if gamma.size == 1:
        gamma = np.full(dk, gamma[0])
    k, v, q = _f64(k).reshape(-1), _f64(v).reshape(-1), _f64(q).reshape(-1)
    o = np.empty(dv)
    lib().kdao_unified_step(dk, dv, _dp(S), _dp(gamma), float(alpha_w), float(beta_w), _dp(k),
                            _dp(v), _dp(q), _dp(o))
    return o


def _threads(nthreads):
    if nthreads is None or nthreads <= 0:
        try:
            return len(os.sched_getaffinity(0))
        except AttributeError:  # pragma: no cover
            return os.cpu_count() or 1
    return nthreads


def forward(params: Params, q, k, v, g_raw, b_raw, A_log, dt_bias, cu_seqlens, pool, state_idx,
            inter=False, heads=None, nthreads=1, chunk_size=None):
    """Run the oracle over packed varlen sequences.

    Returns ``(out, pool_after, inter_states)``; ``pool_after`` is a fp64 copy of the pool with
    the final states written (prefill/decode) or unchanged (verify), ``inter_states`` is the
    [T][H][dv][dk] per-token state buffer when ``inter`` is true.  ``heads`` restricts the
    computation to a subset of heads (other heads' outputs are left as NaN).  With
    ``chunk_size`` set, the chunk closed form is used instead of the token recurrence.
    Work is split over heads across ``nthreads`` threads (the C call releases the GIL).
    """
    L = lib()
    q, k, v = _f64(q), _f64(k), _f64(v)
    g_raw, b_raw, A_log = _f64(g_raw), _f64(b_raw), _f64(A_log)
    dt_bias = _f64(dt_bias)
    cu = _i32(cu_seqlens)
    sidx = _i32(state_idx)
    pool = _f64(pool).copy()
    T = q.shape[0]
    H, dv, dk = params.num_heads, params.dv, params.dk
    out = np.full((T, H, dv), np.nan)
    inter_buf = np.full((T, H, dv, dk), np.nan) if inter else None
    heads = list(range(H)) if heads is None else sorted(int(h) for h in heads)
    nseq = len(sidx)
    nslots = pool.shape[0]

    def run(h):
        if chunk_size is None:
            rc = L.kdao_forward(ctypes.byref(params), _dp(q), _dp(k), _dp(v), _dp(g_raw),
                                _dp(b_raw), _dp(A_log), _dp(dt_bias), _ip(cu), nseq, _dp(pool),
                                nslots, _ip(sidx), _dp(out), _dp(inter_buf), h, h + 1)
        else:
            rc = L.kdao_chunk_forward(ctypes.byref(params), int(chunk_size), _dp(q), _dp(k), _dp(v),
                                      _dp(g_raw), _dp(b_raw), _dp(A_log), _dp(dt_bias), _ip(cu),
                                      nseq, _dp(pool), nslots, _ip(sidx), _dp(out), h, h + 1)
        if rc != 0:
            raise ValueError(f"oracle rejected its arguments (status {rc})")

    n = min(_threads(nthreads), len(heads))
    if n <= 1:
        for h in heads:
            run(h)
    else:
        with ThreadPoolExecutor(max_workers=n) as ex:
            list(ex.map(run, heads))
    return out, pool, inter_buf
