"""KDA state as explicit products of per-token transition matrices (fp64).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py). Independent of the two C
forms: it never applies a rank-one update in place. Each token's step is the
affine map S -> M_t S + B_t with the dense K x K transition

    M_t = (I - beta_t k_t k_t^T) Diag(exp(g_t)),    B_t = beta_t k_t v_t^T,

so the state after token t is the unrolled sum

    S_t = (M_t ... M_1) S_0 + sum_{u<=t} (M_t ... M_{u+1}) B_u,

and o_t = scale * S_t^T q_t. Meant for a handful of tokens (each product is
a dense K x K matrix).
"""
from __future__ import annotations

import numpy as np


def _arr(x):
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def unrolled(q, k, v, g, beta, initial_state=None, scale=None):
    """One sequence: q, k, g [T, H, K]; v [T, H, V]; beta [T, H];
    initial_state [H, K, V] or None. Returns (o [T, H, V], S_T [H, K, V])."""
    q, k, v, g, beta = (_arr(t) for t in (q, k, v, g, beta))
    T, H, K = q.shape
    V = v.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(K)
    s0 = np.zeros((H, K, V)) if initial_state is None else _arr(initial_state)
    o = np.zeros((T, H, V))
    fin = np.zeros((H, K, V))
    eye = np.eye(K)
    for h in range(H):
        M = [(eye - beta[t, h] * np.outer(k[t, h], k[t, h])) @ np.diag(np.exp(g[t, h]))
             for t in range(T)]
        B = [beta[t, h] * np.outer(k[t, h], v[t, h]) for t in range(T)]
        S = s0[h]
        for t in range(T):
            # (M_t ... M_1) S_0
            prod = eye
            for u in range(t, -1, -1):
                prod = prod @ M[u]
            St = prod @ s0[h]
            # + sum_u (M_t ... M_{u+1}) B_u
            for u in range(t + 1):
                tail = eye
                for w in range(t, u, -1):
                    tail = tail @ M[w]
                St = St + tail @ B[u]
            o[t, h] = scale * (St.T @ q[t, h])
            S = St
        fin[h] = S
    return o, fin
