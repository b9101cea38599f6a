"""kda_chunk_prefill_noalloc through the C ABI, against the fp64 oracle.

The allocation-free entry point serves callers that may not allocate device
memory (a host framework that owns every allocation, a serving loop that
must stay out of the driver's allocator, a sandboxed plug-in). It uses a
fixed scratch array inside the library instead of a workspace. Two calls in
a row, on different inputs and sharing that array, must each match the
oracle within the parity bar of the other GPU tests (and agree with the
allocating entry point), an oversized call must be refused before anything
runs, a host pointer must be refused like the allocating entry point
refuses it, and bad cu_seqlens contents must be reported by
kda_last_device_error(). This file is collected last so that a run stopping
at the first failure has run every other test already.
"""
import numpy as np
import pytest
import torch

import kda_inputs as KI
import prefill_kda_chunk_gb300 as K

pytestmark = pytest.mark.gpu

REL_L2 = 1e-2
MAX_ABS = 2e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from prefill_kda_chunk_gb300 import build
    build.build()
    K.lib()


def _args(x, packed, out, fin, scale):
    T, H = x["q"].shape[0], x["q"].shape[1]
    N = x["cu_seqlens"].numel() - 1 if packed else 1
    return (x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(), x["g"].data_ptr(),
            x["beta"].data_ptr(),
            0 if x["initial_state"] is None else x["initial_state"].data_ptr(),
            x["cu_seqlens"].data_ptr() if packed else 0, 1, T, H, 128, 128, N, scale,
            out.data_ptr(), fin.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _dev(d):
    x = {n: d[n].cuda() for n in ("q", "k", "v", "g", "beta", "cu_seqlens")}
    x["initial_state"] = None if d["initial_state"] is None else d["initial_state"].cuda()
    return x


def _run(fn, d, packed):
    x = _dev(d)
    N = x["cu_seqlens"].numel() - 1 if packed else 1
    out = torch.full_like(x["v"], float("nan"))
    fin = torch.full((N, x["q"].shape[1], 128, 128), float("nan"), device="cuda")
    rc = fn(*_args(x, packed, out, fin, d["scale"]))
    assert rc == 0, K.STATUS.get(rc, rc)
    rc = K.kda_last_device_error(torch.cuda.current_stream().cuda_stream)
    assert rc == 0, K.STATUS.get(rc, rc)
    return out, fin


def _close(a, b):
    a = a.double().cpu().numpy()
    b = np.asarray(b, dtype=np.float64)
    assert np.isfinite(a).all()
    rel = np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)
    mx = np.abs(a - b).max() / max(np.abs(b).max(), 1e-300)
    assert rel <= REL_L2 and mx <= MAX_ABS, (rel, mx)


def _oracle(d):
    import oracle
    return oracle.recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"],
                            initial_state=d["initial_state"], cu_seqlens=d["cu_seqlens"],
                            scale=d["scale"])


def test_noalloc_matches_oracle_two_calls():
    cases = [(KI.make_case([100, 7, 33], H=3, seed=31, init_state=True), True),
             (KI.make_case([250], H=4, seed=32, init_state=False), False)]
    for d, packed in cases:  # two calls in a row on the shared scratch
        o_na, f_na = _run(K.kda_chunk_prefill_noalloc, d, packed)
        o_ref, f_ref = _oracle(d)
        _close(o_na, o_ref)
        _close(f_na, f_ref)
        # and the same result as the allocating entry point, within the same bar
        o_al, f_al = _run(K.kda_chunk_prefill, d, packed)
        _close(o_na, o_al.double().cpu().numpy())
        _close(f_na, f_al.double().cpu().numpy())


def test_noalloc_strong_decay_matches_oracle():
    """Strong decay in both of its forms: a packed batch with one head at -9
    per token (factored about the middle of each chunk's decay range) and one
    at -12 (the exact form, whose list lives in the fixed scratch too)."""
    d = KI.make_case([90, 40, 130], H=3, seed=33, init_state=True)
    d["g"][:, 0, :] = -9.0
    d["g"][:, 1, :] = -12.0
    o_na, f_na = _run(K.kda_chunk_prefill_noalloc, d, True)
    o_ref, f_ref = _oracle(d)
    _close(o_na, o_ref)
    _close(f_na, f_ref)


def test_noalloc_rejects_oversized_call():
    # 8192 tokens x 64 heads: 512 chunks x 64 heads x 17408 B of chunk records
    # (~570 MB, all held at once by this entry point), above the 64 MiB array
    assert 512 * 64 * 17408 > (64 << 20)
    dummy = torch.empty(16, dtype=torch.float32, device="cuda")
    p = dummy.data_ptr()
    rc = K.kda_chunk_prefill_noalloc(p, p, p, p, p, 0, 0, 1, 8192, 64, 128, 128, 1, 1.0, p, 0,
                                     torch.cuda.current_stream().cuda_stream)
    assert rc == K.STATUS_CODE["KDA_ERR_SCRATCH_LIMIT"]


def test_noalloc_rejects_host_pointer():
    """A pageable host buffer in place of q is refused before any launch."""
    d = KI.make_case([40], H=2, seed=34)
    x = _dev(d)
    out = torch.full_like(x["v"], float("nan"))
    fin = torch.full((1, 2, 128, 128), float("nan"), device="cuda")
    q_host = d["q"].contiguous()          # CPU tensor
    args = list(_args(x, False, out, fin, d["scale"]))
    args[0] = q_host.data_ptr()
    rc = K.kda_chunk_prefill_noalloc(*args)
    assert rc == K.STATUS_CODE["KDA_ERR_NOT_DEVICE_MEMORY"]
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all() and torch.isnan(fin).all()


def test_noalloc_bad_cu_seqlens_reported():
    """Decreasing cu_seqlens: the kernels skip all work, the call returns
    KDA_OK (the check is on the device) and kda_last_device_error() reports
    KDA_ERR_BAD_CU_SEQLENS once, then KDA_OK."""
    d = KI.make_case([20, 30, 14], H=2, seed=35, init_state=True)
    x = _dev(d)
    x["cu_seqlens"] = torch.tensor([0, 30, 20, 64], dtype=torch.int32, device="cuda")
    out = torch.full_like(x["v"], float("nan"))
    fin = torch.full((3, 2, 128, 128), float("nan"), device="cuda")
    rc = K.kda_chunk_prefill_noalloc(*_args(x, True, out, fin, d["scale"]))
    assert rc == 0
    s = torch.cuda.current_stream().cuda_stream
    assert K.kda_last_device_error(s) == K.STATUS_CODE["KDA_ERR_BAD_CU_SEQLENS"]
    assert K.kda_last_device_error(s) == 0
    assert torch.isnan(out.float()).all() and torch.isnan(fin).all()
    # the shared array is usable again right after
    d2 = KI.make_case([33, 9], H=2, seed=36, init_state=True)
    o, f = _run(K.kda_chunk_prefill_noalloc, d2, True)
    o_ref, f_ref = _oracle(d2)
    _close(o, o_ref)
    _close(f, f_ref)
