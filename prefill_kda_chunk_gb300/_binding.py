"""ctypes binding of libkda_gb300.so (include/kda.h).

Argument marshalling only: every step of the prefill runs in the library's
CUDA kernels. PyTorch supplies device memory and the current stream. There
is no fallback: if the library is missing or the device is not sm_103, calls
raise.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libkda_gb300.so")

STATUS = {
    0: "KDA_OK", -1: "KDA_ERR_NULL_ARG", -2: "KDA_ERR_BAD_SHAPE", -3: "KDA_ERR_UNSUPPORTED_DIM",
    -4: "KDA_ERR_MISALIGNED", -5: "KDA_ERR_BAD_CU_SEQLENS", -6: "KDA_ERR_CUDA",
    -7: "KDA_ERR_DEVICE_TIMEOUT", -8: "KDA_ERR_NO_DEVICE_SUPPORT", -9: "KDA_ERR_ALIAS",
    -10: "KDA_ERR_GATE_RANGE", -11: "KDA_ERR_CAPTURE", -12: "KDA_ERR_WRONG_DEVICE",
    -13: "KDA_ERR_NOT_DEVICE_MEMORY", -14: "KDA_ERR_SCRATCH_LIMIT", -15: "KDA_ERR_BAD_FLAGS",
}
# input preprocessing flags (include/kda.h)
PRE_NORM_QK = 1
PRE_GATE_LOGITS = 2
STATUS_CODE = {v: k for k, v in STATUS.items()}

_lib = None
_lock = threading.Lock()


class KdaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        self.name = STATUS.get(code, str(code))
        super().__init__(f"{where}: {self.name} ({kda_status_string(code)})")


def lib() -> ctypes.CDLL:
    """Load the library (once). Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(
                    f"{LIB_PATH} is missing; build it with "
                    "`python -m prefill_kda_chunk_gb300.build`")
            L = ctypes.CDLL(LIB_PATH)
            vp, i64, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float
            L.kda_chunk_prefill.restype = ctypes.c_int
            L.kda_chunk_prefill.argtypes = [vp] * 7 + [i64] * 6 + [f32, vp, vp, vp]
            L.kda_chunk_prefill_ex.restype = ctypes.c_int
            L.kda_chunk_prefill_ex.argtypes = [vp] * 7 + [i64] * 6 + [f32, ctypes.c_int, vp, vp, vp]
            L.kda_chunk_prefill_noalloc.restype = ctypes.c_int
            L.kda_chunk_prefill_noalloc.argtypes = [vp] * 7 + [i64] * 6 + [f32, vp, vp, vp]
            L.kda_decode_step.restype = ctypes.c_int
            L.kda_decode_step.argtypes = [vp] * 7 + [i64] * 4 + [f32, ctypes.c_int, vp, vp]
            L.kda_backward_workspace_bytes.restype = ctypes.c_int64
            L.kda_backward_workspace_bytes.argtypes = [i64] * 4 + [ctypes.c_int]
            L.kda_chunk_prefill_backward.restype = ctypes.c_int
            L.kda_chunk_prefill_backward.argtypes = [vp] * 7 + [i64] * 6 + [f32] + [vp] * 9
            L.kda_status_string.restype = ctypes.c_char_p
            L.kda_status_string.argtypes = [ctypes.c_int]
            L.kda_last_device_error.restype = ctypes.c_int
            L.kda_last_device_error.argtypes = [vp]
            L.kda_workspace_release.restype = ctypes.c_int
            L.kda_workspace_release.argtypes = []
            L.kda_workspace_bytes.restype = i64
            L.kda_workspace_bytes.argtypes = [i64, i64, i64, i64, ctypes.c_int]
            L.kda_stage_timing_begin.restype = ctypes.c_int
            L.kda_stage_timing_begin.argtypes = [ctypes.c_int]
            L.kda_stage_timing_end.restype = ctypes.c_int
            L.kda_stage_timing_end.argtypes = [ctypes.POINTER(ctypes.c_double),
                                               ctypes.POINTER(ctypes.c_double),
                                               ctypes.POINTER(ctypes.c_int)]
            L.kda_set_recurrent_impl.restype = ctypes.c_int
            L.kda_set_recurrent_impl.argtypes = [ctypes.c_int]
            L.kda_set_scan_segments.restype = ctypes.c_int
            L.kda_set_scan_segments.argtypes = [ctypes.c_int]
            L.kda_set_backward_impl.restype = ctypes.c_int
            L.kda_set_backward_impl.argtypes = [ctypes.c_int]
            L.kda_test_stall_recurrent.restype = ctypes.c_int
            L.kda_test_stall_recurrent.argtypes = [ctypes.c_int, i64]
            L.kda_build_info.restype = ctypes.c_char_p
            L.kda_build_info.argtypes = []
            _lib = L
    return _lib


# ------------------------------------------------------------ raw C calls

def kda_chunk_prefill(q, k, v, g, beta, initial_state, cu_seqlens, B, T, H, K, V, N, scale,
                      out, final_state, stream) -> int:
    """The C entry point, pointers as ints (0 = NULL). Returns the status."""
    return lib().kda_chunk_prefill(q, k, v, g, beta, initial_state, cu_seqlens, B, T, H, K, V, N,
                                   scale, out, final_state, stream)


def kda_chunk_prefill_ex(q, k, v, g, beta, initial_state, cu_seqlens, B, T, H, K, V, N, scale,
                         flags, out, final_state, stream) -> int:
    """The C entry point with input preprocessing flags (PRE_*)."""
    return lib().kda_chunk_prefill_ex(q, k, v, g, beta, initial_state, cu_seqlens, B, T, H, K, V,
                                      N, scale, flags, out, final_state, stream)


def kda_chunk_prefill_noalloc(q, k, v, g, beta, initial_state, cu_seqlens, B, T, H, K, V, N,
                              scale, out, final_state, stream) -> int:
    """The allocation-free C entry point (fixed 64 MiB scratch inside the
    library), pointers as ints. Returns the status."""
    return lib().kda_chunk_prefill_noalloc(q, k, v, g, beta, initial_state, cu_seqlens, B, T, H,
                                           K, V, N, scale, out, final_state, stream)


def kda_decode_step(q, k, v, g, beta, state_in, state_out, N, H, K, V, scale, flags, out,
                    stream) -> int:
    """The one-token decode C entry point, pointers as ints (0 = NULL)."""
    return lib().kda_decode_step(q, k, v, g, beta, state_in, state_out, N, H, K, V, scale, flags,
                                 out, stream)


def kda_backward_workspace_bytes(B, T, H, N, has_cu_seqlens) -> int:
    """Workspace bytes of a gradient call with these sizes (0 on bad sizes)."""
    return lib().kda_backward_workspace_bytes(B, T, H, N, int(bool(has_cu_seqlens)))


def kda_chunk_prefill_backward(q, k, v, g, beta, initial_state, cu_seqlens, B, T, H, K, V, N,
                               scale, d_out, d_final_state, dq, dk, dv, dg, dbeta,
                               d_initial_state, stream) -> int:
    """The gradient C entry point, pointers as ints (0 = NULL)."""
    return lib().kda_chunk_prefill_backward(q, k, v, g, beta, initial_state, cu_seqlens, B, T, H,
                                            K, V, N, scale, d_out, d_final_state, dq, dk, dv, dg,
                                            dbeta, d_initial_state, stream)


def kda_status_string(code: int) -> str:
    return lib().kda_status_string(int(code)).decode()


def kda_last_device_error(stream=0) -> int:
    return lib().kda_last_device_error(stream)


def kda_workspace_release() -> int:
    return lib().kda_workspace_release()


def kda_workspace_bytes(B, T, H, N, has_cu_seqlens) -> int:
    return lib().kda_workspace_bytes(B, T, H, N, int(bool(has_cu_seqlens)))


def kda_stage_timing_begin(max_calls: int) -> int:
    return lib().kda_stage_timing_begin(int(max_calls))


def kda_stage_timing_end():
    """Returns (status, intra_ms_mean, recurrent_ms_mean, calls)."""
    a, b, n = ctypes.c_double(), ctypes.c_double(), ctypes.c_int()
    rc = lib().kda_stage_timing_end(ctypes.byref(a), ctypes.byref(b), ctypes.byref(n))
    return rc, a.value, b.value, n.value


def kda_set_recurrent_impl(impl: int) -> int:
    """1 = 16-token chunks (default), 3 = 64-token chunks on tcgen05 (two
    kernels), 4 = 64-token chunks in one cooperative launch."""
    return lib().kda_set_recurrent_impl(int(impl))


def kda_set_scan_segments(segments: int) -> int:
    """Segment-parallel scan for fixed-length calls: 0 = automatic, 1 = off,
    P >= 2 = P segments per sequence."""
    return lib().kda_set_scan_segments(int(segments))


def kda_set_backward_impl(impl: int) -> int:
    """Gradients: 0 = chunked (default), 1 = token-serial."""
    return lib().kda_set_backward_impl(int(impl))


def kda_test_stall_recurrent(chunk: int, wait_ns: int = 0) -> int:
    """Test hook: the recurrent kernel's record producer stops before `chunk`
    and its waits give up after `wait_ns` (-1: off)."""
    return lib().kda_test_stall_recurrent(int(chunk), int(wait_ns))


def kda_build_info() -> str:
    return lib().kda_build_info().decode()


# ------------------------------------------------------------ torch front

def _ptr(t):
    return 0 if t is None else t.data_ptr()


def _flags(normalize_qk, gate_logits):
    return (PRE_NORM_QK if normalize_qk else 0) | (PRE_GATE_LOGITS if gate_logits else 0)


def chunk_prefill(q, k, v, g, beta, initial_state=None, cu_seqlens=None, scale=None, out=None,
                  final_state=None, output_final_state=True, stream=None, normalize_qk=False,
                  gate_logits=False):
    """Chunked KDA prefill on the current CUDA device.

    q, k, v: bf16 [T, H, 128] (packed or one sequence) or [B, T, H, 128];
    g: fp32 like q; beta: fp32 [..., H]; initial_state: fp32 [N, H, 128, 128]
    or None; cu_seqlens: int32 [N+1] on the device or None. Returns
    (o, final_state) with o bf16 like v and final_state fp32 [N, H, 128, 128]
    (None if output_final_state is False and final_state is None).
    normalize_qk / gate_logits: q, k are raw projections to be L2-normalised,
    and g holds gate logits whose logsigmoid is the log decay (done in the
    kernels).
    """
    import torch

    if q.dim() == 4:
        B, T, H, K = q.shape
    elif q.dim() == 3:
        B, (T, H, K) = 1, q.shape
    else:
        raise ValueError("q must be [T, H, K] or [B, T, H, K]")
    V = v.shape[-1]
    if cu_seqlens is not None:
        if B != 1:
            raise ValueError("cu_seqlens needs B == 1")
        if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda:
            raise ValueError("cu_seqlens must be an int32 CUDA tensor")
        N = cu_seqlens.numel() - 1
    else:
        N = B
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16),
                        ("v", v, torch.bfloat16), ("g", g, torch.float32),
                        ("beta", beta, torch.float32)):
        if t.dtype != dt:
            raise ValueError(f"{name} must be {dt}")
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if k.shape != q.shape or g.shape != q.shape or v.shape[:-1] != q.shape[:-1]:
        raise ValueError("q, k, g must share a shape and v must match it but for the last dim")
    if tuple(beta.shape) != tuple(q.shape[:-1]):
        raise ValueError("beta must be q.shape[:-1]")
    if initial_state is not None:
        if initial_state.dtype != torch.float32 or not initial_state.is_contiguous():
            raise ValueError("initial_state must be a contiguous fp32 tensor")
        if tuple(initial_state.shape) != (N, H, K, V):
            raise ValueError(f"initial_state must be [{N}, {H}, {K}, {V}]")
    if scale is None:
        scale = 1.0 / math.sqrt(K)
    if out is None:
        out = torch.empty_like(v)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, K, V), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    flags = _flags(normalize_qk, gate_logits)
    if flags:
        rc = kda_chunk_prefill_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                  _ptr(initial_state), _ptr(cu_seqlens), B, T, H, K, V, N,
                                  float(scale), flags, _ptr(out), _ptr(final_state), stream)
    else:
        rc = kda_chunk_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                               _ptr(initial_state), _ptr(cu_seqlens), B, T, H, K, V, N,
                               float(scale), _ptr(out), _ptr(final_state), stream)
    if rc != 0:
        raise KdaError(rc, "kda_chunk_prefill")
    return out, final_state


def decode_step(q, k, v, g, beta, state=None, scale=None, out=None, state_out=None,
                in_place=False, stream=None, normalize_qk=False, gate_logits=False):
    """One decode token per sequence on the current CUDA device.

    q, k, v: bf16 [N, H, 128]; g: fp32 [N, H, 128]; beta: fp32 [N, H];
    state: fp32 [N, H, 128, 128] or None (zero state). Returns (o, new_state).
    With in_place=True the new state is written over `state`. normalize_qk /
    gate_logits as for chunk_prefill.
    """
    import torch

    if q.dim() != 3:
        raise ValueError("q must be [N, H, K]")
    N, H, K = q.shape
    V = v.shape[-1]
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16),
                        ("v", v, torch.bfloat16), ("g", g, torch.float32),
                        ("beta", beta, torch.float32)):
        if t.dtype != dt:
            raise ValueError(f"{name} must be {dt}")
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if k.shape != q.shape or g.shape != q.shape or v.shape[:-1] != q.shape[:-1]:
        raise ValueError("q, k, g must share a shape and v must match it but for the last dim")
    if tuple(beta.shape) != (N, H):
        raise ValueError("beta must be [N, H]")
    if state is not None:
        if state.dtype != torch.float32 or not state.is_contiguous():
            raise ValueError("state must be a contiguous fp32 tensor")
        if tuple(state.shape) != (N, H, K, V):
            raise ValueError(f"state must be [{N}, {H}, {K}, {V}]")
    if in_place:
        if state is None:
            raise ValueError("in_place needs a state")
        state_out = state
    elif state_out is None:
        state_out = torch.empty((N, H, K, V), dtype=torch.float32, device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(K)
    if out is None:
        out = torch.empty_like(v)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    rc = kda_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state),
                         _ptr(state_out), N, H, K, V, float(scale),
                         _flags(normalize_qk, gate_logits), _ptr(out), stream)
    if rc != 0:
        raise KdaError(rc, "kda_decode_step")
    return out, state_out


def chunk_prefill_backward(q, k, v, g, beta, d_out, initial_state=None, cu_seqlens=None,
                           scale=None, d_final_state=None, d_initial_state=True, stream=None):
    """Gradients of ``chunk_prefill`` on the current CUDA device.

    Inputs as for chunk_prefill (no preprocessing flags), plus d_out (bf16,
    like v: dL/do) and d_final_state (fp32 [N, H, 128, 128] or None = 0).
    Returns (dq, dk, dv, dg, dbeta, d_initial_state), fp32, shaped like q, k,
    v, g, beta and [N, H, 128, 128]; d_initial_state is None when asked for
    with False.
    """
    import torch

    if q.dim() == 4:
        B, T, H, K = q.shape
    elif q.dim() == 3:
        B, (T, H, K) = 1, q.shape
    else:
        raise ValueError("q must be [T, H, K] or [B, T, H, K]")
    V = v.shape[-1]
    if cu_seqlens is not None:
        if B != 1:
            raise ValueError("cu_seqlens needs B == 1")
        if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda:
            raise ValueError("cu_seqlens must be an int32 CUDA tensor")
        N = cu_seqlens.numel() - 1
    else:
        N = B
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16),
                        ("v", v, torch.bfloat16), ("g", g, torch.float32),
                        ("beta", beta, torch.float32), ("d_out", d_out, torch.bfloat16)):
        if t.dtype != dt:
            raise ValueError(f"{name} must be {dt}")
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if k.shape != q.shape or g.shape != q.shape or v.shape[:-1] != q.shape[:-1]:
        raise ValueError("q, k, g must share a shape and v must match it but for the last dim")
    if d_out.shape != v.shape:
        raise ValueError("d_out must be shaped like v")
    if tuple(beta.shape) != tuple(q.shape[:-1]):
        raise ValueError("beta must be q.shape[:-1]")
    for name, t in (("initial_state", initial_state), ("d_final_state", d_final_state)):
        if t is not None:
            if t.dtype != torch.float32 or not t.is_contiguous() or not t.is_cuda:
                raise ValueError(f"{name} must be a contiguous fp32 CUDA tensor")
            if tuple(t.shape) != (N, H, K, V):
                raise ValueError(f"{name} must be [{N}, {H}, {K}, {V}]")
    if scale is None:
        scale = 1.0 / math.sqrt(K)
    f32 = dict(dtype=torch.float32, device=q.device)
    dq, dk, dg = (torch.empty(q.shape, **f32) for _ in range(3))
    dv = torch.empty(v.shape, **f32)
    dbeta = torch.empty(beta.shape, **f32)
    ds0 = torch.empty((N, H, K, V), **f32) if d_initial_state else None
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    rc = kda_chunk_prefill_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                    _ptr(initial_state), _ptr(cu_seqlens), B, T, H, K, V, N,
                                    float(scale), _ptr(d_out), _ptr(d_final_state), _ptr(dq),
                                    _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta), _ptr(ds0), stream)
    if rc != 0:
        raise KdaError(rc, "kda_chunk_prefill_backward")
    return dq, dk, dv, dg, dbeta, ds0


def check_device_error(stream=None):
    """Synchronise the stream and raise if a kernel recorded an error."""
    import torch

    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    rc = kda_last_device_error(stream)
    if rc != 0:
        raise KdaError(rc, "device")
