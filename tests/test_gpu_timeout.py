"""A bounded device wait that runs out is reported and leaves the context usable.

The recurrent kernel's test hook (kda_test_stall_recurrent) stops every
record producer before a chosen chunk and shortens both roles' wait limit.
The consumers' wait for that chunk then ends after the limit: they record
KDA_ERR_DEVICE_TIMEOUT in the device error word and leave. Nothing faults
or traps, every copy that was issued completes before its CTA exits, and the
next call without the hook must match the oracle.
"""
import numpy as np
import pytest
import torch

import kda_inputs as KI
import prefill_kda_chunk_gb300 as K

pytestmark = pytest.mark.gpu

KDA_ERR_DEVICE_TIMEOUT = -7


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from prefill_kda_chunk_gb300 import build
    build.build()
    K.lib()


def call(d, x):
    return K.chunk_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"],
                           initial_state=x["initial_state"], cu_seqlens=x["cu_seqlens"],
                           scale=d["scale"])


def test_recurrent_wait_runs_out_then_clean_call():
    import oracle
    # sequences of 19, 3, 0 and 13 chunks: the stall before chunk 5 hits the
    # first and last, the second finishes before it
    d = KI.make_case([300, 37, 0, 200], H=2, seed=123, init_state=True)
    x = {n: d[n].cuda().contiguous() for n in ("q", "k", "v", "g", "beta")}
    x["initial_state"] = d["initial_state"].cuda()
    x["cu_seqlens"] = d["cu_seqlens"].cuda()
    stream = torch.cuda.current_stream().cuda_stream
    assert K.kda_set_recurrent_impl(1) == 0
    assert K.kda_last_device_error(stream) == 0
    assert K.kda_test_stall_recurrent(5, 5_000_000) == 0       # waits give up after 5 ms
    try:
        call(d, x)
        rc = K.kda_last_device_error(stream)
    finally:
        assert K.kda_test_stall_recurrent(-1) == 0
    assert rc == KDA_ERR_DEVICE_TIMEOUT
    assert K.kda_last_device_error(stream) == 0                 # the read cleared the word
    # the context still works and the next call is right
    o, f = call(d, x)
    K.check_device_error()
    o_ref, f_ref = oracle.recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                    initial_state=d["initial_state"],
                                    cu_seqlens=d["cu_seqlens"], scale=d["scale"])
    for got, ref in ((o, o_ref), (f, f_ref)):
        got = got.double().cpu().numpy()
        assert np.isfinite(got).all()
        assert np.linalg.norm(got - ref) / np.linalg.norm(ref) < 1e-2
        assert np.max(np.abs(got - ref)) < 2e-2 * np.max(np.abs(ref))


def test_stall_hook_arguments():
    assert K.kda_test_stall_recurrent(-2, 0) != 0
    assert K.kda_test_stall_recurrent(3, -1) != 0
    assert K.kda_test_stall_recurrent(-1, 0) == 0
