"""Gradients of KDA prefill in the chunk-wise WY form (fp64, numpy).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py). It is the reverse mode of
the chunk algebra that the GPU prefill uses ("Kimi K3 的三個系統設計",
section "為什麼 FlashKDA 選擇 16-token chunks": a token-parallel part per
16-token chunk and a recurrent part over the chunks), written out step by
step with exact per-pair exponentials and no blocking, and checked against
the token-level reverse pass (kda_backward.c). It is the plan of a chunked
GPU backward: one reverse chain over the chunks plus chunk-parallel work.

Forward, per sequence and head, for chunk n with S the state entering it
(rows r, i = 0..L-1 of the chunk, G_r = sum_{u<=r} g_u per key channel):

    A[r,i] = beta_r sum_c k_rc k_ic e^(G_rc - G_ic)      (i < r)
    P[r,i] = scale sum_c q_rc k_ic e^(G_rc - G_ic)       (i <= r)
    T  = (I + A)^-1,  M = T diag(beta)
    W  = M (K e^G),   Ut = M V
    Qg = scale Q e^G, Kd = K e^(G_L - G), gamma = e^(G_L)
    U  = Ut - W S,  O = Qg S + P U,  S_next = Diag(gamma) S + Kd^T U

Reverse, given dO and dS_next:

    dU = P^T dO + Kd dS_next
    dS = Diag(gamma) dS_next + Qg^T dO - W^T dU          (to the chunk before)
    dQg = dO S^T, dP = tril(dO U^T), dKd = U dS_next^T
    dgamma = rowsum(dS_next o S), dW = -dU S^T, dUt = dU

then through the WY construction (dM = dUt V^T + dW (K e^G)^T, dT = dM
diag(beta), dA = -T^T dT T^T on the strict lower triangle) and the gated
products to dq, dk, dv, dbeta and dG, and dg as the reverse cumulative sum
of dG within the chunk.
"""
from __future__ import annotations

import numpy as np


def _arr(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def _chunk_forward(q, k, v, g, b, S, scale):
    """The chunk's WY quantities (exact pairwise exponentials) and outputs."""
    L, K = k.shape
    G = np.cumsum(g, axis=0)                                    # [L, K]
    E = np.exp(G[:, None, :] - G[None, :, :])                   # [r, i, c]; used for i <= r
    low = np.tril(np.ones((L, L)), -1)
    lowd = np.tril(np.ones((L, L)))
    A = b[:, None] * np.einsum("rc,ic,ric->ri", k, k, np.where(low[..., None] > 0, E, 0.0)) * low
    P = scale * np.einsum("rc,ic,ric->ri", q, k, np.where(lowd[..., None] > 0, E, 0.0)) * lowd
    T = np.linalg.inv(np.eye(L) + A)
    M = T * b[None, :]
    eG = np.exp(G)
    Kg = k * eG
    W = M @ Kg
    Ut = M @ v
    Qg = scale * q * eG
    Kd = k * np.exp(G[-1][None, :] - G)
    gam = np.exp(G[-1])
    U = Ut - W @ S
    O = Qg @ S + P @ U
    S_next = gam[:, None] * S + Kd.T @ U
    return dict(G=G, E=E, low=low, lowd=lowd, A=A, P=P, T=T, M=M, eG=eG, Kg=Kg, W=W, Ut=Ut,
                Qg=Qg, Kd=Kd, gam=gam, U=U, O=O, S_next=S_next)


def _chunk_backward(q, k, v, g, b, S, scale, f, dO, dSn):
    """Reverse of _chunk_forward. Returns (dq, dk, dv, dg, dbeta, dS)."""
    L, K = k.shape
    P, Kd, W, Qg, U, T, M = f["P"], f["Kd"], f["W"], f["Qg"], f["U"], f["T"], f["M"]
    E, low, lowd, G = f["E"], f["low"], f["lowd"], f["G"]
    # the recurrent part
    dU = P.T @ dO + Kd @ dSn
    dS = f["gam"][:, None] * dSn + Qg.T @ dO - W.T @ dU
    dQg = dO @ S.T
    dP = (dO @ U.T) * lowd
    dKd = U @ dSn.T
    dgam = np.sum(dSn * S, axis=1)
    dW = -dU @ S.T
    dUt = dU
    # the WY construction
    dM = dUt @ v.T + dW @ f["Kg"].T
    dv = M.T @ dUt
    dKg = M.T @ dW
    dT = dM * b[None, :]
    db = np.sum(dM * T, axis=0)                                  # M[r,i] = T[r,i] beta_i
    dA = -(T.T @ dT @ T.T) * low
    dq = np.zeros((L, K))
    dk = np.zeros((L, K))
    dG = np.zeros((L, K))
    # A[r,i] = beta_r sum_c k_rc k_ic E[r,i,c]
    Am = np.where(low[..., None] > 0, E, 0.0)                    # [r, i, c]
    db += np.einsum("ri,rc,ic,ric->r", dA, k, k, Am)
    wA = (dA * b[:, None])[..., None] * Am                       # beta_r dA[r,i] E[r,i,c]
    dk += np.einsum("ric,ic->rc", wA, k)
    dk += np.einsum("ric,rc->ic", wA, k)
    tA = wA * k[:, None, :] * k[None, :, :]
    dG += tA.sum(axis=1)
    dG -= tA.sum(axis=0)
    # P[r,i] = scale sum_c q_rc k_ic E[r,i,c]
    Pm = np.where(lowd[..., None] > 0, E, 0.0)
    wP = (scale * dP)[..., None] * Pm
    dq += np.einsum("ric,ic->rc", wP, k)
    dk += np.einsum("ric,rc->ic", wP, q)
    tP = wP * q[:, None, :] * k[None, :, :]
    dG += tP.sum(axis=1)
    dG -= tP.sum(axis=0)
    # Qg = scale q e^G;  Kd = k e^(G_L - G);  gamma = e^(G_L);  Kg = k e^G
    dq += scale * dQg * f["eG"]
    dG += dQg * Qg
    dk += dKd * np.exp(G[-1][None, :] - G)
    dG -= dKd * Kd
    dG[-1] += np.sum(dKd * Kd, axis=0) + dgam * f["gam"]
    dk += dKg * f["eG"]
    dG += dKg * f["Kg"]
    # G_r = sum_{u<=r} g_u
    dg = np.cumsum(dG[::-1], axis=0)[::-1]
    return dq, dk, dv, dg, db, dS


def chunked_backward(q, k, v, g, beta, dout, initial_state=None, d_final_state=None,
                     cu_seqlens=None, scale=None, chunk=16):
    """Same arguments and result keys as ``oracle.recurrent_backward``."""
    q, k, v, g, beta, dout = (_arr(t) for t in (q, k, v, g, beta, dout))
    T, H, K = q.shape
    V = v.shape[2]
    cu = [0, T] if cu_seqlens is None else [int(c) for c in _arr(cu_seqlens)]
    N = len(cu) - 1
    s0 = _arr(initial_state)
    dsf = _arr(d_final_state)
    if scale is None:
        scale = 1.0 / np.sqrt(K)
    out = {"o": np.zeros((T, H, V)), "final_state": np.zeros((N, H, K, V)),
           "dq": np.zeros((T, H, K)), "dk": np.zeros((T, H, K)), "dv": np.zeros((T, H, V)),
           "dg": np.zeros((T, H, K)), "dbeta": np.zeros((T, H)),
           "d_initial_state": np.zeros((N, H, K, V))}
    for n in range(N):
        spans = [(a, min(a + chunk, cu[n + 1])) for a in range(cu[n], cu[n + 1], chunk)]
        for h in range(H):
            S = np.zeros((K, V)) if s0 is None else s0[n, h].copy()
            states, fwd = [], []
            for a, e in spans:
                f = _chunk_forward(q[a:e, h], k[a:e, h], v[a:e, h], g[a:e, h], beta[a:e, h], S,
                                   scale)
                states.append(S)
                fwd.append(f)
                out["o"][a:e, h] = f["O"]
                S = f["S_next"]
            out["final_state"][n, h] = S
            dS = np.zeros((K, V)) if dsf is None else dsf[n, h].copy()
            for (a, e), S_in, f in reversed(list(zip(spans, states, fwd))):
                dq, dk, dv, dg, db, dS = _chunk_backward(q[a:e, h], k[a:e, h], v[a:e, h],
                                                         g[a:e, h], beta[a:e, h], S_in, scale,
                                                         f, dout[a:e, h], dS)
                out["dq"][a:e, h], out["dk"][a:e, h], out["dv"][a:e, h] = dq, dk, dv
                out["dg"][a:e, h], out["dbeta"][a:e, h] = dg, db
            out["d_initial_state"][n, h] = dS
    return out
