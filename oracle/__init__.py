"""fp64 CPU oracle for chunked KDA prefill.

TEST INFRASTRUCTURE ONLY. The test suite, the package's smoke check and the
benchmark's CPU-baseline leg may import this; the CUDA library and its Python
binding never do, and the two share no code (only the seeded input module
``kda_inputs`` serves both).

Three independently written forms of the same result:

* ``recurrent`` -- the token-by-token recurrence (kda_recurrent.c), the
  definition every other form is checked against;
* ``chunked`` -- the chunk-wise WY form with exact per-pair exponentials
  (kda_chunked.c), the algebra the GPU kernels use, written without blocking
  or factoring;
* ``unrolled`` (unrolled.py) -- the state written out as explicit products of
  per-token transition matrices, for a handful of tokens;
* ``segment_scan`` (segment_scan.py) -- the chunks of a sequence cut into
  segments, each reduced to one affine state map on its own, combined
  serially, then replayed (the segment-parallel form for long sequences).

And the gradients of the same map: ``recurrent_backward`` (kda_backward.c),
the reverse pass of the token recurrence written line by line, pinned by
central differences of its own forward pass; and ``chunked_backward``
(chunked_backward.py), the reverse pass of the chunk-wise WY form, checked
against it.

What is computed: Kimi Delta Attention keeps a fixed-size recurrent state per
head that each new token updates ("Kimi K3 開源基礎設施", section "FlashKDA";
"Kimi K3 的三個系統設計", section "第一個設計"). The update is the gated
delta rule with a per-channel decay on the key rows,

    S_t = (I - beta_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + beta_t k_t v_t^T,
    o_t = scale * S_t^T q_t,

with S a K x V fp64 matrix (row = key channel). The chunked form cuts each
sequence into 16-token chunks ("Kimi K3 的三個系統設計", section
"為什麼 FlashKDA 選擇 16-token chunks").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_SOURCES = ["kda_recurrent.c", "kda_chunked.c", "kda_backward.c"]
_lib = None
_lock = threading.Lock()

from .unrolled import unrolled  # noqa: E402  (pure numpy, no build needed)
from .chunked_backward import chunked_backward  # noqa: E402  (pure numpy)
from .segment_scan import segment_scan  # noqa: E402  (pure numpy)


def build(force: bool = False) -> str:
    """Compile the C oracle into oracle/_build/liboracle.so (gcc, no GPU)."""
    srcs = [os.path.join(_HERE, s) for s in _SOURCES]
    if not force and os.path.exists(_LIB_PATH):
        newest = max(os.path.getmtime(s) for s in srcs)
        if os.path.getmtime(_LIB_PATH) >= newest:
            return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
           "-o", tmp] + srcs + ["-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            f64p = ctypes.POINTER(ctypes.c_double)
            f32p = ctypes.POINTER(ctypes.c_float)
            i64p = ctypes.POINTER(ctypes.c_int64)
            i64 = ctypes.c_int64
            lib.kda_oracle_recurrent.restype = ctypes.c_int
            lib.kda_oracle_recurrent.argtypes = [f32p] * 5 + [f64p, i64p] + [i64] * 4 + [
                ctypes.c_double, f64p, i64, f64p, ctypes.c_int, ctypes.c_int, ctypes.c_int]
            lib.kda_oracle_chunked.restype = ctypes.c_int
            lib.kda_oracle_chunked.argtypes = [f32p] * 5 + [f64p, i64p] + [i64] * 5 + [
                ctypes.c_double, f64p, i64, f64p, ctypes.c_int]
            lib.kda_oracle_backward.restype = ctypes.c_int
            lib.kda_oracle_backward.argtypes = [f64p] * 6 + [i64p] + [i64] * 4 + [
                ctypes.c_double] + [f64p] * 10 + [ctypes.c_int, ctypes.c_int]
            _lib = lib
    return _lib


def _f32(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor (bf16 promotes to fp32 exactly)
        x = x.detach().to("cpu").float().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a, ct):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ct))


def _prep(q, k, v, g, beta, initial_state, cu_seqlens):
    q, k, v, g, beta = (_f32(t) for t in (q, k, v, g, beta))
    if q.ndim != 3 or k.shape != q.shape or g.shape != q.shape:
        raise ValueError("q, k, g must be [T, H, K]")
    T, H, K = q.shape
    if v.ndim != 3 or v.shape[:2] != (T, H):
        raise ValueError("v must be [T, H, V]")
    V = v.shape[2]
    if beta.shape != (T, H):
        raise ValueError("beta must be [T, H]")
    if cu_seqlens is None:
        cu = np.array([0, T], dtype=np.int64)
    else:
        if hasattr(cu_seqlens, "detach"):
            cu_seqlens = cu_seqlens.detach().cpu().numpy()
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
        if cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
            raise ValueError("cu_seqlens must start at 0, end at T and not decrease")
    N = len(cu) - 1
    s0 = _f64(initial_state)
    if s0 is not None and s0.shape != (N, H, K, V):
        raise ValueError("initial_state must be [N, H, K, V]")
    return q, k, v, g, beta, s0, cu, T, H, K, V, N


def recurrent(q, k, v, g, beta, initial_state=None, cu_seqlens=None, scale=None,
              out_tokens=None, threads=0, mutation=0, normalize_qk=False, gate_logits=False):
    """Token-by-token fp64 recurrence. Returns (o [T, H, V], final [N, H, K, V])
    as float64 numpy arrays; o rows at or past ``out_tokens`` are left zero.

    ``normalize_qk``: q and k are raw and are divided by sqrt(sum x^2 + 1e-6)
    per (token, head) before use. ``gate_logits``: g holds gate logits x and
    the log decay is logsigmoid(x). Both are done in fp64 inside the oracle.

    ``mutation`` plants a known mistake (see kda_recurrent.c); only the pin
    tests use it, to show that each pin catches what it should."""
    q, k, v, g, beta, s0, cu, T, H, K, V, N = _prep(q, k, v, g, beta, initial_state, cu_seqlens)
    if scale is None:
        scale = 1.0 / np.sqrt(K)
    ot = T if out_tokens is None else int(out_tokens)
    o = np.zeros((max(ot, 0), H, V), dtype=np.float64)
    fs = np.zeros((N, H, K, V), dtype=np.float64)
    rc = _load().kda_oracle_recurrent(
        _ptr(q, ctypes.c_float), _ptr(k, ctypes.c_float), _ptr(v, ctypes.c_float),
        _ptr(g, ctypes.c_float), _ptr(beta, ctypes.c_float), _ptr(s0, ctypes.c_double),
        _ptr(cu, ctypes.c_int64), N, H, K, V, float(scale), _ptr(o, ctypes.c_double), ot,
        _ptr(fs, ctypes.c_double), int(threads),
        (1 if normalize_qk else 0) | (2 if gate_logits else 0), int(mutation))
    if rc:
        raise RuntimeError(f"kda_oracle_recurrent failed ({rc})")
    return o, fs


def chunked(q, k, v, g, beta, initial_state=None, cu_seqlens=None, scale=None,
            out_tokens=None, threads=0, chunk=16):
    """Chunk-wise WY form in fp64 (exact per-pair exponentials). Same return
    as ``recurrent``."""
    q, k, v, g, beta, s0, cu, T, H, K, V, N = _prep(q, k, v, g, beta, initial_state, cu_seqlens)
    if scale is None:
        scale = 1.0 / np.sqrt(K)
    ot = T if out_tokens is None else int(out_tokens)
    o = np.zeros((max(ot, 0), H, V), dtype=np.float64)
    fs = np.zeros((N, H, K, V), dtype=np.float64)
    rc = _load().kda_oracle_chunked(
        _ptr(q, ctypes.c_float), _ptr(k, ctypes.c_float), _ptr(v, ctypes.c_float),
        _ptr(g, ctypes.c_float), _ptr(beta, ctypes.c_float), _ptr(s0, ctypes.c_double),
        _ptr(cu, ctypes.c_int64), N, H, K, V, int(chunk), float(scale),
        _ptr(o, ctypes.c_double), ot, _ptr(fs, ctypes.c_double), int(threads))
    if rc:
        raise RuntimeError(f"kda_oracle_chunked failed ({rc})")
    return o, fs


def recurrent_backward(q, k, v, g, beta, dout, initial_state=None, d_final_state=None,
                       cu_seqlens=None, scale=None, threads=0, mutation=0):
    """Gradients of the token recurrence in fp64 (kda_backward.c), for the
    loss L with dL/do = ``dout`` [T, H, V] and dL/d(final state) =
    ``d_final_state`` [N, H, K, V] (None: 0). Inputs are taken as given, in
    float64 (bf16 and fp32 values convert exactly).

    Returns a dict of float64 numpy arrays: dq, dk, dg [T, H, K]; dv [T, H, V];
    dbeta [T, H]; d_initial_state [N, H, K, V]; and the forward results o
    [T, H, V] and final_state [N, H, K, V] of the same pass.

    ``threads``: host threads over the (sequence, head) pairs (0 = every
    core; the results do not depend on it). ``mutation`` plants a known
    mistake in the reverse pass (see kda_backward.c); only the pin tests use
    it."""
    q, k, v, g, beta, dout = (_f64(t) for t in (q, k, v, g, beta, dout))
    if q.ndim != 3 or k.shape != q.shape or g.shape != q.shape:
        raise ValueError("q, k, g must be [T, H, K]")
    T, H, K = q.shape
    if v.ndim != 3 or v.shape[:2] != (T, H) or dout.shape != v.shape:
        raise ValueError("v and dout must be [T, H, V]")
    V = v.shape[2]
    if beta.shape != (T, H):
        raise ValueError("beta must be [T, H]")
    if cu_seqlens is None:
        cu = np.array([0, T], dtype=np.int64)
    else:
        if hasattr(cu_seqlens, "detach"):
            cu_seqlens = cu_seqlens.detach().cpu().numpy()
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
        if cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
            raise ValueError("cu_seqlens must start at 0, end at T and not decrease")
    N = len(cu) - 1
    s0, dsf = _f64(initial_state), _f64(d_final_state)
    for name, x in (("initial_state", s0), ("d_final_state", dsf)):
        if x is not None and x.shape != (N, H, K, V):
            raise ValueError(f"{name} must be [N, H, K, V]")
    if scale is None:
        scale = 1.0 / np.sqrt(K)
    out = {"o": np.zeros((T, H, V)), "final_state": np.zeros((N, H, K, V)),
           "dq": np.zeros((T, H, K)), "dk": np.zeros((T, H, K)), "dv": np.zeros((T, H, V)),
           "dg": np.zeros((T, H, K)), "dbeta": np.zeros((T, H)),
           "d_initial_state": np.zeros((N, H, K, V))}
    d = ctypes.c_double
    rc = _load().kda_oracle_backward(
        _ptr(q, d), _ptr(k, d), _ptr(v, d), _ptr(g, d), _ptr(beta, d), _ptr(s0, d),
        _ptr(cu, ctypes.c_int64), N, H, K, V, float(scale), _ptr(dout, d), _ptr(dsf, d),
        _ptr(out["o"], d), _ptr(out["final_state"], d), _ptr(out["dq"], d), _ptr(out["dk"], d),
        _ptr(out["dv"], d), _ptr(out["dg"], d), _ptr(out["dbeta"], d),
        _ptr(out["d_initial_state"], d), int(threads), int(mutation))
    if rc:
        raise RuntimeError(f"kda_oracle_backward failed ({rc})")
    return out


__all__ = ["build", "recurrent", "chunked", "unrolled", "recurrent_backward", "chunked_backward",
           "segment_scan"]
