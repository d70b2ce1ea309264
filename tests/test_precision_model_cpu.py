"""Numerics models (CPU only), evaluated in fp64 with every operand rounded where the kernels round
it and compared with the oracle's token recurrence on the same inputs: the bf16 tensor-core
prefill, and the ring of the buffered decode.

Rounding points of the kernels (bf16 inputs, d = 128, chunk 64):
  * alpha, beta, k_hat, q_hat in fp32;
  * the off-diagonal 16 x 16 blocks of A and P from fp16 operands (keys decayed to the start of
    the row block, rows decayed from it), the diagonal blocks in fp32; A and P kept in fp32;
  * U and W by block forward substitution, X_I = T_II B_I - sum_{J<I} F_IJ X_J, every MMA operand
    rounded to tf32 (round to nearest), T_II and F_IJ formed in fp32;
  * the record in fp16 (W, Q_bar, K_tilde, P, U), e^{G_L} in fp32;
  * the state pass as one MMA per chunk, Delta_{i+1} = U_{i+1} - W'_{i+1} S_i - Z_{i+1} Delta_i
    with W' = W Diag(e^{G_L} of chunk i) and Z = W K_tilde_i^T as fp16 images, S and Delta as fp16
    operands, fp32 accumulation and an fp32 master state.

The model must meet the 2e-3 bound of bf16 inputs; the same model with bf16 operands in place of
fp16 must not, which is why the record and the state-pass operands are fp16 (same 11-bit
significand as tf32, every value far inside fp16 range).  The recurrence is "linear_attention",
section "KDA：逐通道的遗忘门"; the chunk form is that page's "矩阵（并行）形式" applied per chunk as
in "两种计算形态"."""
import math

import numpy as np
import pytest
import torch

import oracle
from kda_gated_delta_gb300 import workloads


def f32(x):
    return np.asarray(x, np.float64).astype(np.float32).astype(np.float64)


def f16(x):
    return np.asarray(x, np.float64).astype(np.float32).astype(np.float16).astype(np.float64)


def bf16(x):
    return torch.from_numpy(np.asarray(x, np.float64)).to(torch.bfloat16).double().numpy()


def tf32(x):
    """fp32 rounded to nearest at 10 fraction bits (ties away from zero, as cvt.rna.tf32)."""
    a = np.asarray(x, np.float64).astype(np.float32)
    b = a.view(np.uint32).astype(np.uint64)
    b = ((b + 0x1000) & 0xFFFFE000).astype(np.uint32)
    return b.view(np.float32).astype(np.float64)


def model(inp, H, D, C, opnd):
    """Outputs [T][H][D] and final pool of the modelled kernels; `opnd` rounds the fp16 operands."""
    q, k, v = (inp[n].double().numpy() for n in ("q", "k", "v"))
    g_raw, b_raw = inp["g_raw"].double().numpy(), inp["b_raw"].double().numpy()
    A_log, dtb = inp["A_log"].double().numpy(), inp["dt_bias"].double().numpy()
    cu, sidx = inp["cu_seqlens"].numpy(), inp["state_idx"].numpy()
    pool = inp["pool"].double().numpy().copy()
    out = np.zeros((q.shape[0], H, D))
    nb = C // 16
    for s in range(len(cu) - 1):
        t_begin, t_end = int(cu[s]), int(cu[s + 1])
        for h in range(H):
            S = pool[sidx[s], h].T.copy()                 # S[c][j], fp32 master state
            rate = math.exp(A_log[h])
            prev = None
            for t0 in range(t_begin, t_end, C):
                L = min(C, t_end - t0)
                x = g_raw[t0:t0 + L, h] + dtb[h]
                sp = np.where(x > 20.0, x, np.log1p(np.exp(np.minimum(x, 20.0))))
                alpha = f32(np.exp(-rate * sp))
                G = np.cumsum(np.log(np.maximum(alpha, 1e-300)), axis=0)
                beta = f32(1.0 / (1.0 + np.exp(-b_raw[t0:t0 + L, h])))
                kk, qq, vv = k[t0:t0 + L, h], q[t0:t0 + L, h], v[t0:t0 + L, h]
                kh = f32(kk / np.sqrt((kk * kk).sum(1, keepdims=True) + 1e-6))
                qh = f32(qq / np.sqrt((qq * qq).sum(1, keepdims=True) + 1e-6) / math.sqrt(D))
                # A (strictly lower) and P (lower with diagonal), zero-padded to C rows
                A = np.zeros((C, C))
                P = np.zeros((C, C))
                for I in range(nb):
                    ri = np.arange(16 * I, min(16 * I + 16, L))
                    if ri.size == 0:
                        continue
                    # diagonal block: fp32 CUDA-core products
                    for J in range(I + 1):
                        rj = np.arange(16 * J, min(16 * J + 16, L))
                        if J == I:
                            dec = np.exp(np.minimum(G[ri][:, None, :] - G[rj][None, :, :], 0.0))   # r >= j kept
                            a_ = np.einsum("rc,jc,rjc->rj", kh[ri], kh[rj], dec)
                            p_ = np.einsum("rc,jc,rjc->rj", qh[ri], kh[rj], dec)
                        else:
                            ref = 16 * I - 1                   # decay split at the row block's start
                            left = opnd(kh[rj] * np.exp(G[ref] - G[rj]))
                            a_ = opnd(kh[ri] * np.exp(G[ri] - G[ref])) @ left.T
                            p_ = opnd(qh[ri] * np.exp(G[ri] - G[ref])) @ left.T
                        A[np.ix_(ri, rj)] = beta[ri][:, None] * a_
                        P[np.ix_(ri, rj)] = p_
                A = f32(np.tril(A, -1))
                P = f32(np.tril(P))
                # U, W by block forward substitution with tf32 operands
                eG = np.exp(G)
                B = np.zeros((C, 2 * D))
                B[:L, :D] = beta[:, None] * vv
                B[:L, D:] = beta[:, None] * kh * eG
                B = tf32(B)
                X = []
                Tii = [f32(np.linalg.inv(np.eye(16) + A[16 * i:16 * i + 16, 16 * i:16 * i + 16])) for i in range(nb)]
                for I in range(nb):
                    acc = tf32(Tii[I]) @ B[16 * I:16 * I + 16]
                    for J in range(I):
                        F = f32(Tii[I] @ A[16 * I:16 * I + 16, 16 * J:16 * J + 16])
                        acc = acc - tf32(F) @ tf32(X[J])
                    X.append(f32(acc))
                Xa = np.concatenate(X, 0)[:L]
                U, W = Xa[:, :D], Xa[:, D:]
                # the record
                Wr, Ur = opnd(W), opnd(U)
                Qr = opnd(qh * eG)
                Kr = opnd(kh * np.exp(G[L - 1][None, :] - G))
                Pr = opnd(P[:L, :L])
                gL = f32(np.exp(G[L - 1]))
                # the state pass: one MMA per chunk on the chain
                So = opnd(S)
                if prev is None:
                    Dl = Ur - Wr @ So
                else:
                    gl_p, Kr_p, Do_p, So_p = prev
                    Wp = opnd(W * gl_p[None, :])
                    Z = opnd(Wr @ Kr_p.T)
                    Dl = Ur - Wp @ So_p - Z @ Do_p
                Do = opnd(f32(Dl))
                out[t0:t0 + L, h] = f32(Qr @ So + Pr @ Do)
                prev = (gL, Kr, Do, So)
                S = f32(gL[:, None] * S + Kr.T @ Do)
            pool[sidx[s], h] = S.T
    return out, pool


def _rel(a, b):
    return float(np.abs(a - b).max() / np.abs(b).max())


CASES = {"workload gates": {}, "mild gates": dict(g_mean=-8.0, g_std=2.0),
         "strong gates": dict(g_mean=4.0, g_std=2.0)}


@pytest.fixture(scope="module")
def runs():
    H, D, C = 4, 128, 64
    res = {}
    for name, kw in CASES.items():
        inp = workloads.make_inputs([700, 333], H, D, torch.bfloat16, pool_slots=4, pool_std=0.01, seed=7, **kw)
        p = oracle.make_params(H, D)
        o_ref, p_ref, _ = oracle.forward(p, inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["b_raw"], inp["A_log"],
                                         inp["dt_bias"], inp["cu_seqlens"], inp["pool"], inp["state_idx"])
        res[name] = (inp, o_ref, p_ref)
    return H, D, C, res


@pytest.mark.parametrize("name", sorted(CASES))
def test_fp16_operands_meet_the_bf16_bound(runs, name):
    H, D, C, res = runs
    inp, o_ref, p_ref = res[name]
    o, pl = model(inp, H, D, C, f16)
    used = inp["state_idx"].numpy()
    e_o, e_s = _rel(o, o_ref), _rel(pl[used], p_ref[used])
    print(f"{name}: fp16 operands, output {e_o:.2e}, state {e_s:.2e}")
    assert e_o <= 2e-3 and e_s <= 2e-3, (e_o, e_s)


@pytest.mark.parametrize("name", sorted(CASES))
def test_bf16_operands_would_not(runs, name):
    """The same model with bf16 operands (8-bit significand) misses the bound: the precision of
    the record and the state-pass operands is a requirement."""
    H, D, C, res = runs
    inp, o_ref, p_ref = res[name]
    o, pl = model(inp, H, D, C, bf16)
    used = inp["state_idx"].numpy()
    e = max(_rel(o, o_ref), _rel(pl[used], p_ref[used]))
    print(f"{name}: bf16 operands, {e:.2e}")
    assert e > 2e-3, e


def replay_model(inp, H, D, L, steps, B, ring_round):
    """The buffered decode (ReplaySSM, sections 3.9-3.12) over `steps` tokens per request: each step
    rebuilds S' from the checkpoint and the ring entries (d_j, k_hat_j, a_j) committed since, takes
    the step, and either appends (d, k_hat, a) to the ring or, when the ring is full or at the last
    step, writes the checkpoint.  `ring_round` rounds the stored d."""
    q, k, v = (inp[n].double().numpy() for n in ("q", "k", "v"))
    g_raw, b_raw = inp["g_raw"].double().numpy(), inp["b_raw"].double().numpy()
    A_log, dtb = inp["A_log"].double().numpy(), inp["dt_bias"].double().numpy()
    sidx = inp["state_idx"].numpy()
    pool = inp["pool"].double().numpy().copy()
    out = np.zeros((B * steps, H, D))
    for b in range(B):
        for h in range(H):
            S0 = pool[sidx[b], h].T.copy()
            ring = []
            rate = math.exp(A_log[h])
            for t in range(steps):
                row = b * steps + t
                x = g_raw[row, h] + dtb[h]
                a = f32(np.exp(-rate * np.where(x > 20.0, x, np.log1p(np.exp(np.minimum(x, 20.0))))))
                beta = f32(1.0 / (1.0 + np.exp(-b_raw[row, h])))
                kk, qq = k[row, h], q[row, h]
                kh = f32(kk / math.sqrt(kk @ kk + 1e-6))
                qh = f32(qq / math.sqrt(qq @ qq + 1e-6) / math.sqrt(D))
                Sr = S0.copy()
                for d_j, k_j, a_j in ring:
                    Sr = a_j[:, None] * Sr + np.outer(k_j, d_j)
                Sd = a[:, None] * Sr
                delta = beta * (v[row, h] - kh @ Sd)
                S_t = Sd + np.outer(kh, delta)
                out[row, h] = f32(qh @ S_t)
                if len(ring) == L - 1 or t == steps - 1:
                    S0, ring = f32(S_t), []
                else:
                    ring.append((ring_round(delta), kh, a))
            pool[sidx[b], h] = S0.T
    return out, pool


def test_buffered_decode_ring_precision():
    """Ring length 16, 6 requests x 4 heads, 33 steps: with fp32 ring entries the model matches the
    oracle to rounding; with bf16 deltas (the state dtype some deployments choose) the error they
    add alone is over a quarter of the 2e-3 bound, which is why the kernel keeps the ring in fp32."""
    H, D, L, B, steps = 4, 128, 16, 6, 33
    inp = workloads.make_inputs([steps] * B, H, D, torch.bfloat16, pool_slots=8, pool_std=0.05, seed=82,
                                dt_bias_std=0.3)
    p = oracle.make_params(H, D)
    o_ref, p_ref, _ = oracle.forward(p, inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["b_raw"], inp["A_log"],
                                     inp["dt_bias"], inp["cu_seqlens"], inp["pool"], inp["state_idx"])
    used = inp["state_idx"].numpy()
    errs = {}
    for name, rnd in (("fp32", f32), ("bf16", bf16)):
        o, pl = replay_model(inp, H, D, L, steps, B, rnd)
        errs[name] = max(_rel(o, o_ref), _rel(pl[used], p_ref[used]))
    print(f"buffered decode ring: fp32 {errs['fp32']:.2e}, bf16 {errs['bf16']:.2e}")
    assert errs["fp32"] <= 1e-5
    assert errs["bf16"] > 5e-4


def test_tf32_operands_cannot_meet_the_fp32_bound():
    """fp32 inputs are held to 1e-5. The same chunk algorithm with tf32 operands (rounded to
    nearest) lands near 1e-3, two orders above that, which is why fp32 inputs run on the fp32
    CUDA-core pair instead of the tensor cores."""
    H, D, C = 2, 128, 64
    inp = workloads.make_inputs([300, 77], H, D, torch.float32, pool_slots=2, pool_std=0.01, seed=8)
    p = oracle.make_params(H, D)
    o_ref, p_ref, _ = oracle.forward(p, inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["b_raw"], inp["A_log"],
                                     inp["dt_bias"], inp["cu_seqlens"], inp["pool"], inp["state_idx"])
    o, pl = model(inp, H, D, C, tf32)
    used = inp["state_idx"].numpy()
    e = max(_rel(o, o_ref), _rel(pl[used], p_ref[used]))
    print(f"fp32 inputs, tf32 operands: {e:.2e}")
    assert e > 1e-4, e
