"""One-token decode step against the fp64 oracle, through the C ABI.

A decode batch of N sequences is the token recurrence with one token per
sequence: the oracle runs it as a packed batch with cu_seqlens = 0, 1, ..., N.
Same bar as the prefill: relative L2 error <= 1e-2 and max abs error
<= 2e-2 * max|ref|, for o and the new state separately.
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


def oracle_step(d, state):
    import oracle
    return oracle.recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"], initial_state=state,
                            cu_seqlens=d["cu_seqlens"], scale=d["scale"])


def check(x, ref, tag):
    x = x.detach().double().cpu().numpy()
    assert np.isfinite(x).all(), tag
    rel = np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300)
    mx = np.max(np.abs(x - ref)) / max(np.max(np.abs(ref)), 1e-300)
    assert rel <= REL_L2 and mx <= MAX_ABS, f"{tag}: rel {rel:.2e} max {mx:.2e}"


def decode_inputs(N, H, seed, init=True, mu=3.0):
    d = KI.make_case([1] * N, H=H, seed=seed, init_state=init, mu=mu)
    x = {n: d[n].cuda().contiguous() for n in ("q", "k", "v", "g", "beta")}
    s0 = None if d["initial_state"] is None else d["initial_state"].cuda()
    return d, x, s0


@pytest.mark.parametrize("N,H,init", [(1, 1, True), (37, 3, True), (5, 8, False), (256, 4, True)])
def test_decode_parity(N, H, init):
    d, x, s0 = decode_inputs(N, H, seed=40 + N, init=init)
    out = torch.full_like(x["v"], float("nan"))
    new = torch.full((N, H, 128, 128), float("nan"), device="cuda")
    o, s1 = K.decode_step(x["q"], x["k"], x["v"], x["g"], x["beta"], state=s0, scale=d["scale"],
                          out=out, state_out=new)
    torch.cuda.synchronize()
    o_ref, s_ref = oracle_step(d, d["initial_state"])
    check(o, o_ref, "o")
    check(s1, s_ref, "state")
    if s0 is not None:
        assert torch.equal(s0.cpu(), d["initial_state"]), "the input state was modified"


def test_decode_in_place_matches_out_of_place_bitwise():
    d, x, s0 = decode_inputs(19, 4, seed=7)
    o1, s1 = K.decode_step(x["q"], x["k"], x["v"], x["g"], x["beta"], state=s0)
    st = s0.clone()
    o2, s2 = K.decode_step(x["q"], x["k"], x["v"], x["g"], x["beta"], state=st, in_place=True)
    torch.cuda.synchronize()
    assert s2.data_ptr() == st.data_ptr()
    assert torch.equal(o1, o2) and torch.equal(s1, st)


def test_decode_steps_follow_the_recurrence():
    """Five decode steps in a row equal the token recurrence over five tokens
    per sequence (o of every step and the final state)."""
    N, H, steps = 6, 2, 5
    d = KI.make_case([steps] * N, H=H, seed=11, init_state=True)
    o_ref, s_ref = oracle_step(d, d["initial_state"])
    # token t of sequence n sits at packed row n * steps + t
    rows = lambda t: torch.arange(N) * steps + t
    state = d["initial_state"].cuda()
    for t in range(steps):
        r = rows(t)
        xs = {n: d[n][r].cuda().contiguous() for n in ("q", "k", "v", "g", "beta")}
        o, state = K.decode_step(xs["q"], xs["k"], xs["v"], xs["g"], xs["beta"], state=state,
                                 scale=d["scale"])
        check(o, o_ref[r.numpy()], f"o at step {t}")
    torch.cuda.synchronize()
    check(state, s_ref, "final state")


def test_prefill_then_decode():
    """Decoding token T+1 from a prefill's final state equals the recurrence
    over T+1 tokens."""
    T, H = 100, 4
    d = KI.make_case([T + 1], H=H, seed=23, init_state=True)
    o_ref, s_ref = oracle_step(d, d["initial_state"])
    x = {n: d[n][:T].cuda().contiguous() for n in ("q", "k", "v", "g", "beta")}
    _, fin = K.chunk_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"],
                             initial_state=d["initial_state"].cuda(), scale=d["scale"])
    y = {n: d[n][T:].cuda().contiguous() for n in ("q", "k", "v", "g", "beta")}
    o, s1 = K.decode_step(y["q"], y["k"], y["v"], y["g"], y["beta"], state=fin, scale=d["scale"])
    K.check_device_error()
    check(o, o_ref[T:], "o of the decoded token")
    check(s1, s_ref, "state after the decoded token")


def test_decode_extreme_gates_need_no_range_limit():
    """Exponentials are exact per channel: g far below the prefill's factored
    range still decodes correctly (reset to beta k v^T)."""
    d, x, s0 = decode_inputs(8, 2, seed=3)
    g = torch.full_like(x["g"], -1e4)
    d2 = dict(d, g=g.cpu())
    o, s1 = K.decode_step(x["q"], x["k"], x["v"], g, x["beta"], state=s0, scale=d["scale"])
    torch.cuda.synchronize()
    o_ref, s_ref = oracle_step(d2, d["initial_state"])
    check(o, o_ref, "o")
    check(s1, s_ref, "state")


def test_decode_large_batch_sampled():
    """The bench size (256 sequences x 64 heads), checked on sampled
    (sequence, head) units against the oracle."""
    N, H = 256, 64
    d, x, s0 = decode_inputs(N, H, seed=5)
    o, s1 = K.decode_step(x["q"], x["k"], x["v"], x["g"], x["beta"], state=s0, scale=d["scale"])
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    for n in rng.choice(N, size=6, replace=False):
        sub = {key: d[key][n:n + 1] for key in ("q", "k", "v", "g", "beta")}
        sub.update(cu_seqlens=torch.tensor([0, 1], dtype=torch.int32), scale=d["scale"])
        o_ref, s_ref = oracle_step(sub, d["initial_state"][n:n + 1])
        check(o[n:n + 1], o_ref, f"o of sequence {n}")
        check(s1[n:n + 1], s_ref, f"state of sequence {n}")


def test_decode_rejects_host_memory():
    d, x, s0 = decode_inputs(2, 1, seed=1)
    host_state = torch.empty(2, 1, 128, 128).pin_memory()
    out = torch.empty_like(x["v"])
    rc = K.kda_decode_step(x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(),
                           x["g"].data_ptr(), x["beta"].data_ptr(), 0, host_state.data_ptr(),
                           2, 1, 128, 128, 1.0, 0, out.data_ptr(),
                           torch.cuda.current_stream().cuda_stream)
    assert rc == K.STATUS_CODE["KDA_ERR_NOT_DEVICE_MEMORY"]
