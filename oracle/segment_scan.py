"""Segment-parallel form of the KDA state recurrence (fp64, numpy).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py). Over chunks the state map
is affine: with the chunk quantities of the WY form (W, Ut, Kd, gamma; see
chunked_backward.py),

    S_{n+1} = A_n S_n + B_n,   A_n = Diag(gamma_n) - Kd_n^T W_n  (K x K),
                               B_n = Kd_n^T Ut_n                 (K x V).

Cut a sequence's chunks into P segments. Each segment j reduces, on its
own, to one affine map

    M_j = A_{e-1} ... A_s,   c_j = sum_{s<=n<e} A_{e-1} ... A_{n+1} B_n,

so the entry states follow from a short serial combine
S_{s_{j+1}} = M_j S_{s_j} + c_j, after which every segment can be replayed
from its entry state independently. This is the segment-parallel scan for
long sequences (the pages mention million-token contexts: "Kimi K3
開源基礎設施"), written out for checking; the GPU path builds its
two-segment case as the split replay.
"""
from __future__ import annotations

import numpy as np

from .chunked_backward import _arr, _chunk_forward


def segment_scan(q, k, v, g, beta, initial_state=None, cu_seqlens=None, scale=None, chunk=16,
                 segments=2):
    """Same inputs as ``oracle.recurrent``. Returns (o [T, H, V], final
    [N, H, K, V]), with every sequence's chunks cut into ``segments`` nearly
    equal segments whose maps are built independently."""
    q, k, v, g, beta = (_arr(t) for t in (q, k, v, g, beta))
    T, H, K = q.shape
    V = v.shape[2]
    cu = [0, T] if cu_seqlens is None else [int(c) for c in _arr(cu_seqlens)]
    N = len(cu) - 1
    s0 = _arr(initial_state)
    if scale is None:
        scale = 1.0 / np.sqrt(K)
    o = np.zeros((T, H, V))
    fin = np.zeros((N, H, K, V))
    for n in range(N):
        spans = [(a, min(a + chunk, cu[n + 1])) for a in range(cu[n], cu[n + 1], chunk)]
        nseg = max(1, min(segments, len(spans)))
        bounds = np.linspace(0, len(spans), nseg + 1).round().astype(int)
        for h in range(H):
            # the chunk maps; each is built from the chunk's own inputs only
            # (_chunk_forward's state argument does not enter W, Ut, Kd, gamma)
            maps = []
            for a, e in spans:
                f = _chunk_forward(q[a:e, h], k[a:e, h], v[a:e, h], g[a:e, h], beta[a:e, h],
                                   np.zeros((K, V)), scale)
                A = np.diag(f["gam"]) - f["Kd"].T @ f["W"]
                B = f["Kd"].T @ f["Ut"]
                maps.append((A, B))
            # per segment, independently: its composed affine map
            seg = []
            for j in range(nseg):
                M, c = np.eye(K), np.zeros((K, V))
                for A, B in maps[bounds[j]:bounds[j + 1]]:
                    M, c = A @ M, A @ c + B
                seg.append((M, c))
            # serial combine over the segments: their entry states
            S = np.zeros((K, V)) if s0 is None else s0[n, h].copy()
            entry = []
            for M, c in seg:
                entry.append(S)
                S = M @ S + c
            fin[n, h] = S
            # replay every segment from its entry state
            for j in range(nseg):
                Sj = entry[j]
                for a, e in spans[bounds[j]:bounds[j + 1]]:
                    f = _chunk_forward(q[a:e, h], k[a:e, h], v[a:e, h], g[a:e, h],
                                       beta[a:e, h], Sj, scale)
                    o[a:e, h] = f["O"]
                    Sj = f["S_next"]
    return o, fin
