"""Gradients of the prefill (kda_chunk_prefill_backward) against the fp64
gradient oracle, through the C ABI.

Same bar as the forward parity tests, for every output separately: relative
L2 error <= 1e-2 and max abs error <= 2e-2 * max|ref|. dL/do is a seeded
bf16 tensor and dL/d(final state) a seeded fp32 one.
"""
import numpy as np
import pytest
import torch

import kda_inputs as KI
import prefill_kda_chunk_gb300 as K

pytestmark = pytest.mark.gpu

REL_L2 = 1e-2
MAX_ABS = 2e-2
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "d_initial_state")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from prefill_kda_chunk_gb300 import build
    build.build()
    K.lib()


# every test runs with both gradient forms: 0 = chunked (default), 1 = token-serial
@pytest.fixture(autouse=True, params=[0, 1], ids=["chunked", "token_serial"])
def backward_impl(request, built):
    assert K.kda_set_backward_impl(request.param) == 0
    yield request.param
    K.kda_set_backward_impl(0)


def make(seqlens, H, seed, init=True, dsf=True):
    d = KI.make_case(seqlens, H=H, seed=seed, init_state=init)
    gen = torch.Generator().manual_seed(seed + 1000)
    T, N = sum(seqlens), len(seqlens)
    d["dout"] = torch.randn(T, H, 128, generator=gen).to(torch.bfloat16)
    d["dsf"] = (torch.randn(N, H, 128, 128, generator=gen) * 0.1) if dsf else None
    return d


def oracle_grads(d):
    import oracle
    r = oracle.recurrent_backward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["dout"],
                                  initial_state=d["initial_state"], d_final_state=d["dsf"],
                                  cu_seqlens=d["cu_seqlens"], scale=d["scale"])
    return [r[n] for n in NAMES]


def gpu_grads(d, packed=True):
    x = {n: d[n].cuda().contiguous() for n in ("q", "k", "v", "g", "beta", "dout")}
    s0 = None if d["initial_state"] is None else d["initial_state"].cuda()
    dsf = None if d["dsf"] is None else d["dsf"].cuda()
    cu = d["cu_seqlens"].cuda() if packed else None
    if not packed:   # fixed-length batch: [B, T, H, 128]
        B = len(d["seqlens"])
        x = {n: t.view(B, -1, *t.shape[1:]) for n, t in x.items()}
    out = K.chunk_prefill_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["dout"],
                                   initial_state=s0, cu_seqlens=cu, scale=d["scale"],
                                   d_final_state=dsf)
    K.check_device_error()
    return out


def check(x, ref, tag):
    x = x.detach().double().cpu().numpy().reshape(ref.shape)
    assert np.isfinite(x).all(), tag
    if not np.any(ref):
        # an exactly zero gradient (e.g. dg of one token on a zero state): the
        # chunked form reaches it as a sum of terms that cancel, so compare
        # absolutely (the other gradients of these cases are O(1))
        assert np.max(np.abs(x)) <= 1e-5, f"{tag}: max {np.max(np.abs(x)):.2e} against 0"
        return
    rel = np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300)
    mx = np.max(np.abs(x - ref)) / max(np.max(np.abs(ref)), 1e-300)
    assert rel <= REL_L2 and mx <= MAX_ABS, f"{tag}: rel {rel:.2e} max {mx:.2e}"


def check_all(d, got, tag):
    for name, x, ref in zip(NAMES, got, oracle_grads(d)):
        check(x, ref, f"{tag} {name}")


@pytest.mark.parametrize("T", [1, 15, 16, 17, 40])
@pytest.mark.parametrize("init", [False, True])
def test_backward_single_sequence(T, init):
    d = make([T], H=2, seed=T + 10 * init, init=init)
    check_all(d, gpu_grads(d), f"T={T}")


def test_backward_ragged_packed_batch():
    d = make([37, 0, 129, 16, 5], H=3, seed=21)
    check_all(d, gpu_grads(d), "ragged")


def test_backward_fixed_batch():
    d = make([70, 70], H=2, seed=22)
    check_all(d, gpu_grads(d, packed=False), "fixed B=2")


def test_backward_without_final_state_gradient():
    d = make([50], H=2, seed=23, dsf=False)
    check_all(d, gpu_grads(d), "dsf=None")


@pytest.mark.parametrize("gval", [-6.0, -9.0, -12.0, -40.0])
def test_backward_strong_decay(gval):
    """Strong decay in each form of the gated products: -6 and -9 per token
    (a chunk's range of G up to 144) factor about the middle of the range;
    -12 and -40 (ranges of 192 and 640) take the exact per-pair form."""
    d = make([64, 9], H=2, seed=24)
    d["g"] = torch.full_like(d["g"], gval)
    check_all(d, gpu_grads(d), f"g={gval}")


def test_backward_strong_decay_mixed_heads():
    """Heads in all three forms in one call: ordinary gates, -9 per token
    (middle of the range) and -12 (exact)."""
    d = make([100, 37], H=3, seed=25)
    d["g"][:, 1, :] = -9.0
    d["g"][:, 2, :] = -12.0
    check_all(d, gpu_grads(d), "mixed heads")


def test_backward_deterministic():
    """Two calls on the same inputs give bitwise equal gradients. Heads in all
    three forms: the exact-form list is filled by atomic appends, in an order
    that may differ between calls, and every output still has one writer."""
    d = make([200, 77], H=3, seed=31)
    d["g"][:, 1, :] = -9.0
    d["g"][:, 2, :] = -12.0
    a = gpu_grads(d)
    b = gpu_grads(d)
    torch.cuda.synchronize()
    for name, x, y in zip(NAMES, a, b):
        assert torch.equal(x, y), name


def test_backward_zero_tokens_passes_state_gradient():
    d = make([0, 0], H=2, seed=25)
    got = gpu_grads(d)
    torch.cuda.synchronize()
    assert torch.equal(got[5].cpu(), d["dsf"])


def test_backward_longer_sequence():
    """Several hundred tokens in several heads: dS carried over many
    checkpoint segments."""
    d = make([700], H=4, seed=26)
    check_all(d, gpu_grads(d), "T=700")


def test_backward_more_units_than_ctas():
    """320 (sequence, head) units: the persistent kernel's CTAs take several
    each, reusing their state ring (lengths 0..37, some past one segment)."""
    lens = [(7 * i) % 38 for i in range(40)]
    d = make(lens, H=8, seed=29)
    check_all(d, gpu_grads(d), "320 units")


def test_backward_bad_cu_seqlens_flagged():
    d = make([20, 30], H=1, seed=27)
    x = {n: d[n].cuda().contiguous() for n in ("q", "k", "v", "g", "beta", "dout")}
    bad = torch.tensor([0, 35, 30], dtype=torch.int32, device="cuda")
    K.chunk_prefill_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["dout"],
                             cu_seqlens=bad)
    rc = K.kda_last_device_error(torch.cuda.current_stream().cuda_stream)
    assert rc == K.STATUS_CODE["KDA_ERR_BAD_CU_SEQLENS"]


def test_backward_consistent_with_forward_by_directional_derivative():
    """The loss is affine in v (the state is linear in v and the initial
    state), so the GPU forward's L(v + D) - L(v - D) equals <dL/dv, 2 D>
    exactly but for rounding: this ties the two GPU paths together. D is
    the bf16-representable step actually taken."""
    d = make([48], H=1, seed=28, init=True)
    got = gpu_grads(d)
    x = {n: d[n].cuda().contiguous() for n in ("q", "k", "g", "beta")}
    s0 = d["initial_state"].cuda()
    gen = torch.Generator().manual_seed(5)
    step = 0.25 * torch.randn(d["v"].shape, generator=gen)
    vp = (d["v"].float() + step).to(torch.bfloat16)
    vm = (d["v"].float() - step).to(torch.bfloat16)

    def loss(vv):
        o, f = K.chunk_prefill(x["q"], x["k"], vv.cuda(), x["g"], x["beta"],
                               initial_state=s0, scale=d["scale"])
        torch.cuda.synchronize()
        return float((o.double().cpu() * d["dout"].double()).sum()
                     + (f.double().cpu() * d["dsf"].double()).sum())

    diff = loss(vp) - loss(vm)
    an = float((got[2].double().cpu() * (vp.double() - vm.double())).sum())
    assert abs(diff - an) <= 0.03 * max(1.0, abs(an)), (diff, an)


@pytest.mark.parametrize("workload", ["fixed_T8192_H64", "fixed_T8192_H96"])
def test_backward_benchmarked_workload_sampled(workload):
    """The gradient call at the sizes it is timed at (one sequence of 8192
    tokens, 64 or 96 heads), every output checked against the oracle on a
    sample of heads: the heads are independent units, so the oracle runs on
    each sampled head's slice of the inputs alone."""
    d = KI.make_inputs(KI.WORKLOADS[workload])
    T, H = d["q"].shape[0], d["q"].shape[1]
    gen = torch.Generator().manual_seed(4242)
    d["dout"] = torch.randn(T, H, 128, generator=gen).to(torch.bfloat16)
    d["dsf"] = torch.randn(1, H, 128, 128, generator=gen) * 0.1
    got = gpu_grads(d)
    torch.cuda.synchronize()
    got = [t.cpu() for t in got]
    rng = np.random.default_rng(7)
    heads = sorted(int(h) for h in rng.choice(H, size=4, replace=False))
    for h in heads:
        sub = {n: d[n][:, h:h + 1].contiguous() for n in ("q", "k", "v", "g", "beta", "dout")}
        sub["initial_state"] = (None if d["initial_state"] is None
                                else d["initial_state"][:, h:h + 1].contiguous())
        sub["dsf"] = d["dsf"][:, h:h + 1].contiguous()
        sub["cu_seqlens"], sub["scale"] = d["cu_seqlens"], d["scale"]
        for name, x, ref in zip(NAMES, got, oracle_grads(sub)):
            check(x[:, h:h + 1], ref, f"head {h} {name}")


def test_backward_varlen_workload_sampled():
    """The gradient call on the packed workload varlen16_T8192_H64 (16 sequences
    of ragged lengths, initial states), checked against the oracle on sampled
    (sequence, head) units: each unit's slice of the inputs alone, its tokens'
    gradients and its d_initial_state."""
    d = KI.make_inputs(KI.WORKLOADS["varlen16_T8192_H64"])
    T, H = d["q"].shape[0], d["q"].shape[1]
    N = len(d["seqlens"])
    gen = torch.Generator().manual_seed(4343)
    d["dout"] = torch.randn(T, H, 128, generator=gen).to(torch.bfloat16)
    d["dsf"] = torch.randn(N, H, 128, 128, generator=gen) * 0.1
    got = gpu_grads(d)
    torch.cuda.synchronize()
    got = [t.cpu() for t in got]
    cu = d["cu_seqlens"].tolist()
    rng = np.random.default_rng(11)
    units = [(int(n), int(h)) for n, h in zip(rng.choice(N, size=3, replace=False),
                                               rng.choice(H, size=3, replace=False))]
    for n, h in units:
        a, b = cu[n], cu[n + 1]
        sub = {k: d[k][a:b, h:h + 1].contiguous() for k in ("q", "k", "v", "g", "beta", "dout")}
        sub["initial_state"] = d["initial_state"][n:n + 1, h:h + 1].contiguous()
        sub["dsf"] = d["dsf"][n:n + 1, h:h + 1].contiguous()
        sub["cu_seqlens"] = torch.tensor([0, b - a], dtype=torch.int32)
        sub["scale"] = d["scale"]
        refs = oracle_grads(sub)
        for name, x, ref in zip(NAMES[:5], got[:5], refs[:5]):
            check(x[a:b, h:h + 1], ref, f"seq {n} head {h} {name}")
        check(got[5][n:n + 1, h:h + 1], refs[5], f"seq {n} head {h} d_initial_state")
