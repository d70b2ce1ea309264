"""Host-side checks of the C ABI (no GPU needed): libkda.so loads and exports every function that
include/kda.h declares, defaults and status strings, and the argument validation that returns
before any work is enqueued.  Pointers passed here are never dereferenced by the host code."""
import ctypes
import os
import re

import pytest

from kda_gated_delta_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return binding.lib()


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w \*]*?\b(kda_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("kda_chunk_prefill", "kda_recurrent_decode", "kda_recurrent_verify",
              "kda_chunk_prefill_workspace_size", "kda_status_string", "kda_params_init",
              "kda_check_device_errors"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_params_defaults(L):
    p = binding.Params()
    L.kda_params_init(ctypes.byref(p), 32, 128)
    assert (p.num_heads, p.head_dim, p.chunk_size) == (32, 128, 64)
    assert (p.io_dtype, p.out_dtype, p.gate_kind) == (binding.KDA_BF16, binding.KDA_BF16, 0)
    assert p.use_lower_bound == 0 and p.scale == 0.0
    assert p.l2_eps == pytest.approx(1e-6) and p.softplus_threshold == 20.0


def test_status_strings(L):
    for s in (0, -1, -2, -3, -4, -5, -6, 12345):
        assert isinstance(binding.status_string(s), str) and binding.status_string(s)


FAKE = 1 << 20          # 16-byte aligned dummy address, never dereferenced on the host
MIS = FAKE + 4          # misaligned


def _params(**kw):
    p = binding.Params()
    binding.lib().kda_params_init(ctypes.byref(p), kw.pop("H", 4), kw.pop("D", 128))
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def _decode(p, q=FAKE, batch=4, pool=FAKE, out=FAKE):
    return binding.lib().kda_recurrent_decode(ctypes.byref(p) if p is not None else None, q, FAKE, FAKE,
                                              FAKE, FAKE, FAKE, None, batch, pool, 8, FAKE, out, None)


def test_decode_validation(L):
    assert _decode(None) == -1
    assert _decode(_params(), batch=-1) == -1
    assert _decode(_params(D=48)) == -2
    assert _decode(_params(io_dtype=7)) == -2
    assert _decode(_params(), q=MIS) == -3
    assert _decode(_params(), pool=MIS) == -3
    assert _decode(_params(), q=None) == -1
    assert _decode(_params(), batch=0) == 0           # empty batch: nothing enqueued


def test_verify_validation(L):
    p = _params(gate_kind=1)
    f = L.kda_recurrent_verify
    assert f(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 4, 0, FAKE, 8, FAKE, FAKE, FAKE, None) == -1
    assert f(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 4, 17, FAKE, 8, FAKE, FAKE, FAKE, None) == -1
    assert f(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 4, 4, FAKE, 8, FAKE, None, FAKE, None) == -1
    assert f(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 4, 4, FAKE, 8, FAKE, MIS, FAKE, None) == -3
    assert f(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0, 4, FAKE, 8, FAKE, None, FAKE, None) == 0


def test_prefill_validation_and_workspace(L):
    p = _params(D=128, chunk_size=64)
    ws = binding.prefill_workspace_size(p, 8, 16384)
    # one record per (chunk, head), bound ceil(T/C) + N chunks.  bf16 inputs at C = 64, D = 128: the
    # tensor-core pair's fp16 record, five operand images (W, Ktil^T, Qbar, U: 64 x 128; P: 64 x 64)
    # and e^{G_L} in fp32; other shapes: the fp32 record W, Qbar, Ktil, U, P and e^{G_L}.
    nrec = 4 * (16384 // 64 + 8)
    per_tc = 2 * (4 * 64 * 128 + 64 * 64) + 4 * 128
    per_f32 = 4 * ((4 * 64 * 128 + 64 * 64 + 128 + 63) // 64 * 64)
    p.io_dtype = binding.KDA_BF16
    assert binding.prefill_workspace_size(p, 8, 16384) >= per_tc * nrec
    assert binding.prefill_workspace_size(p, 8, 16384) < per_tc * nrec + 64 * 1024
    p.io_dtype = binding.KDA_F32
    assert binding.prefill_workspace_size(p, 8, 16384) >= per_f32 * nrec
    assert ws > 0
    assert binding.prefill_workspace_size(_params(D=48), 8, 100) == 0
    f = L.kda_chunk_prefill

    def call(p, T=100, N=2, ws_ptr=FAKE, ws_bytes=None, cu=FAKE):
        wsb = binding.prefill_workspace_size(p, N, T) if ws_bytes is None else ws_bytes
        return f(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, cu, N, T, FAKE, 8, FAKE, FAKE,
                 ws_ptr, wsb, None)

    assert call(_params(D=128, chunk_size=48)) == -2
    assert call(_params(D=128, gate_kind=1)) == -2             # prefill is built for the per-channel gate
    assert call(p, ws_ptr=None) == -4
    assert call(p, ws_bytes=16) == -4
    assert call(p, ws_ptr=FAKE + 16) == -4                     # workspace must be 256-byte aligned
    assert call(p, cu=None) == -1
    assert call(p, T=0) == 0 and call(p, N=0) == 0
    assert call(p, N=-1) == -1
    assert call(p, T=(1 << 31) - 64, ws_bytes=1 << 40) == -2    # total_tokens limit (kda.h)


def test_selftest_validation(L):
    """The bounded-wait self-test checks its arguments on the host before any CUDA call."""
    f = L.kda_selftest_wait_timeout
    f.restype = ctypes.c_int32
    f.argtypes = [ctypes.c_uint32, ctypes.c_void_p, ctypes.c_void_p]
    assert f(0, None, None) == -1
    assert f((1 << 24) + 1, None, None) == -1
    assert f(8, FAKE + 2, None) == -3


def test_replay_validation(L):
    """kda_replay_decode: ring length in [1, 32], ring buffers and cursors present and aligned."""
    f = L.kda_replay_decode

    def call(p=None, batch=4, ring_len=8, rd=FAKE, rk=FAKE, ra=FAKE, wp=FAKE, out=FAKE):
        p = _params() if p is None else p
        return f(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, batch, FAKE, 8, FAKE,
                 rd, rk, ra, ring_len, wp, None, out, None)

    assert call(ring_len=0) == -1
    assert call(ring_len=33) == -1
    assert call(batch=-1) == -1
    assert call(p=_params(D=48)) == -2
    assert call(rd=None) == -1
    assert call(wp=None) == -1
    assert call(out=None) == -1
    assert call(rk=MIS) == -3
    assert call(ra=MIS) == -3
    assert call(batch=0) == 0


def test_commit_validation(L):
    """kda_commit_verified_states: t_draft in [1, 16], buffers present, 16-byte aligned states."""
    f = L.kda_commit_verified_states
    p = _params()

    def call(p=p, inter=FAKE, batch=4, t_draft=4, acc=FAKE, pool=FAKE):
        return f(ctypes.byref(p) if p is not None else None, inter, batch, t_draft, acc, pool, 8, FAKE, None)

    assert call(p=None) == -1
    assert call(t_draft=0) == -1
    assert call(t_draft=17) == -1
    assert call(batch=-1) == -1
    assert call(p=_params(D=48)) == -2
    assert call(inter=None) == -1
    assert call(acc=None) == -1
    assert call(inter=MIS) == -3
    assert call(pool=MIS) == -3
    assert call(batch=0) == 0


def test_snapshot_and_timed_prefill_validation(L):
    """kda_chunk_prefill_snapshots needs an aligned snapshot buffer and a non-negative capacity;
    kda_chunk_prefill_timed needs KDA_PREFILL_PHASE_EVENTS non-null event handles."""
    p = _params(D=128, chunk_size=64)
    wsb = binding.prefill_workspace_size(p, 2, 100)
    args = (ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 2, 100, FAKE, 8, FAKE, FAKE,
            FAKE, wsb)
    snap = L.kda_chunk_prefill_snapshots
    assert snap(*args, None, 10, None) == -1
    assert snap(*args, FAKE, -1, None) == -1
    assert snap(*args, MIS, 10, None) == -3
    timed = L.kda_chunk_prefill_timed
    assert timed(*args, None, None) == -1
    events = (ctypes.c_void_p * 4)()                            # all null
    assert timed(*args, None, events) == -1
