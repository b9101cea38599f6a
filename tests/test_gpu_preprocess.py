"""Input preprocessing inside the kernels (KDA_PRE_NORM_QK, KDA_PRE_GATE_LOGITS)
against the fp64 oracle doing the same preprocessing, through the C ABI.

Raw projections: q and k rows with norms far from 1, g given as gate logits.
Same bar as the other parity tests: relative L2 <= 1e-2 and max abs
<= 2e-2 * max|ref| for o and the final state separately.
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


def check(x, ref, tag):
    x = x.detach().double().cpu().numpy()
    assert np.isfinite(x).all(), tag
    rel = np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300)
    mx = np.max(np.abs(x - ref)) / max(np.max(np.abs(ref)), 1e-300)
    assert rel <= REL_L2 and mx <= MAX_ABS, f"{tag}: rel {rel:.2e} max {mx:.2e}"


def oracle(d, norm, logits):
    import oracle as O
    return O.recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"],
                       initial_state=d["initial_state"], cu_seqlens=d["cu_seqlens"],
                       scale=d["scale"], normalize_qk=norm, gate_logits=logits)


FLAGS = [(True, True), (True, False), (False, True)]
IDS = ["norm+logits", "norm", "logits"]


@pytest.mark.parametrize("norm,logits", FLAGS, ids=IDS)
@pytest.mark.parametrize("seqlens", [[300], [37, 0, 129, 16, 5]], ids=["one", "ragged"])
def test_prefill_preprocessing(seqlens, norm, logits):
    d = KI.make_raw_case(seqlens, H=3, seed=sum(seqlens) + norm + 2 * logits, init_state=True)
    if not logits:   # plain log decays when the gate is given directly
        d["g"] = torch.nn.functional.logsigmoid(d["g"])
    if not norm:     # then q and k must already be unit rows
        for n in ("q", "k"):
            x = d[n].float()
            d[n] = (x / torch.linalg.vector_norm(x, dim=-1, keepdim=True)).to(torch.bfloat16)
    x = {n: d[n].cuda().contiguous() for n in ("q", "k", "v", "g", "beta")}
    out = torch.full_like(x["v"], float("nan"))
    fin = torch.full((len(seqlens), 3, 128, 128), float("nan"), device="cuda")
    o, f = K.chunk_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"],
                           initial_state=d["initial_state"].cuda(),
                           cu_seqlens=d["cu_seqlens"].cuda(), scale=d["scale"], out=out,
                           final_state=fin, normalize_qk=norm, gate_logits=logits)
    K.check_device_error()
    o_ref, f_ref = oracle(d, norm, logits)
    check(o, o_ref, "o")
    check(f, f_ref, "final_state")


def test_prefill_preprocessing_fixed_batch():
    """cu_seqlens = NULL (B sequences of T tokens) takes the same path."""
    B, T, H = 2, 70, 2
    d = KI.make_raw_case([T] * B, H=H, seed=77)
    x = {n: d[n].cuda().contiguous() for n in ("q", "k", "v", "g", "beta")}
    q4 = {n: t.view(B, T, *t.shape[1:]) for n, t in x.items()}
    o, f = K.chunk_prefill(q4["q"], q4["k"], q4["v"], q4["g"], q4["beta"], scale=d["scale"],
                           normalize_qk=True, gate_logits=True)
    K.check_device_error()
    o_ref, f_ref = oracle(d, True, True)
    check(o.view(B * T, H, 128), o_ref, "o")
    check(f, f_ref, "final_state")


@pytest.mark.parametrize("norm,logits", FLAGS, ids=IDS)
def test_decode_preprocessing(norm, logits):
    N, H = 40, 3
    d = KI.make_raw_case([1] * N, H=H, seed=90 + norm + 2 * logits, init_state=True)
    if not logits:
        d["g"] = torch.nn.functional.logsigmoid(d["g"])
    if not norm:
        for n in ("q", "k"):
            x = d[n].float()
            d[n] = (x / torch.linalg.vector_norm(x, dim=-1, keepdim=True)).to(torch.bfloat16)
    x = {n: d[n].cuda().contiguous() for n in ("q", "k", "v", "g", "beta")}
    o, s1 = K.decode_step(x["q"], x["k"], x["v"], x["g"], x["beta"],
                          state=d["initial_state"].cuda(), scale=d["scale"], normalize_qk=norm,
                          gate_logits=logits)
    torch.cuda.synchronize()
    o_ref, s_ref = oracle(d, norm, logits)
    check(o, o_ref, "o")
    check(s1, s_ref, "state")


def test_preprocessing_equals_preprocessed_inputs():
    """The flags give the same result (to rounding) as handing the kernels
    inputs preprocessed by the caller."""
    d = KI.make_raw_case([200], H=2, seed=3)
    x = {n: d[n].cuda().contiguous() for n in ("q", "k", "v", "g", "beta")}
    o1, f1 = K.chunk_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], scale=d["scale"],
                             normalize_qk=True, gate_logits=True)
    qn = torch.nn.functional.normalize(x["q"].float(), dim=-1, eps=0).to(torch.bfloat16)
    kn = torch.nn.functional.normalize(x["k"].float(), dim=-1, eps=0).to(torch.bfloat16)
    g = torch.nn.functional.logsigmoid(x["g"])
    o2, f2 = K.chunk_prefill(qn, kn, x["v"], g, x["beta"], scale=d["scale"])
    K.check_device_error()
    rel_o = (o1.float() - o2.float()).norm() / o2.float().norm()
    rel_f = (f1 - f2).norm() / f2.norm()
    assert rel_o < 1e-2 and rel_f < 1e-2, (float(rel_o), float(rel_f))


@pytest.mark.parametrize("impl", [1, 3, 4], ids=["c16", "c64_split", "c64_fused"])
def test_preprocessing_with_each_recurrent_kernel(impl):
    """The preprocessing lives in the intra-chunk kernel of each path (the
    16-token one and the 64-token tcgen05 one): check every path."""
    d = KI.make_raw_case([150, 33], H=2, seed=60 + impl, init_state=True)
    x = {n: d[n].cuda().contiguous() for n in ("q", "k", "v", "g", "beta")}
    assert K.kda_set_recurrent_impl(impl) == 0
    try:
        o, f = K.chunk_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"],
                               initial_state=d["initial_state"].cuda(),
                               cu_seqlens=d["cu_seqlens"].cuda(), scale=d["scale"],
                               normalize_qk=True, gate_logits=True)
        K.check_device_error()
    finally:
        K.kda_set_recurrent_impl(1)
    o_ref, f_ref = oracle(d, True, True)
    check(o, o_ref, "o")
    check(f, f_ref, "final_state")


@pytest.mark.parametrize("impl", [1, 3, 4], ids=["c16", "c64_split", "c64_fused"])
@pytest.mark.parametrize("spread", [1.0, 4.0], ids=["middle", "exact"])
def test_preprocessing_strong_decay(impl, spread):
    """Gate logits far below 0. At about -6 per token the 16-token chunks'
    decay ranges (about 96) are factored about their middle; at about -24
    (spread 4) the intra-chunk kernel takes its exact form. Both do the q/k
    normalisation and the logsigmoid themselves."""
    d = KI.make_raw_case([150, 33], H=2, seed=70 + impl, init_state=True, mu=-6.0)
    gen = torch.Generator().manual_seed(71)
    d["g"] = d["g"] * spread + 0.5 * torch.randn(d["g"].shape, generator=gen)
    x = {n: d[n].cuda().contiguous() for n in ("q", "k", "v", "g", "beta")}
    assert K.kda_set_recurrent_impl(impl) == 0
    try:
        o, f = K.chunk_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"],
                               initial_state=d["initial_state"].cuda(),
                               cu_seqlens=d["cu_seqlens"].cuda(), scale=d["scale"],
                               normalize_qk=True, gate_logits=True)
        K.check_device_error()
    finally:
        K.kda_set_recurrent_impl(1)
    o_ref, f_ref = oracle(d, True, True)
    check(o, o_ref, "o")
    check(f, f_ref, "final_state")
