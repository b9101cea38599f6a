"""CUDA path against the fp64 oracle, through the C ABI.

Bar (per tensor, per case): relative L2 error <= 1e-2 and max abs error
<= 2e-2 * max|ref|, for o (bf16) and final_state (fp32) separately.
"""
import math

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


# every test runs on each path: 1 = 16-token chunks (warp-MMA recurrent kernel),
# 3 = 64-token chunks on tcgen05 (two kernels), 4 = 64-token chunks in one
# cooperative launch with an L2 ring of records
@pytest.fixture(autouse=True, params=[1, 3, 4], ids=["c16", "c64_split", "c64_fused"])
def recurrent_impl(request, built):
    assert K.kda_set_recurrent_impl(request.param) == 0
    yield request.param
    K.kda_set_recurrent_impl(1)


def to_dev(d):
    dev = {}
    for key in ("q", "k", "v", "g", "beta"):
        dev[key] = d[key].cuda().contiguous()
    dev["initial_state"] = None if d["initial_state"] is None else d["initial_state"].cuda()
    dev["cu_seqlens"] = d["cu_seqlens"].cuda()
    return dev


def run_gpu(d, packed=True, canary=True, **kw):
    x = to_dev(d)
    N = len(d["seqlens"])
    out = torch.empty_like(x["v"])
    fin = torch.empty((N, x["q"].shape[1], 128, 128), dtype=torch.float32, device="cuda")
    if canary:
        out.fill_(float("nan"))
        fin.fill_(float("nan"))
    o, f = K.chunk_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"],
                           initial_state=x["initial_state"],
                           cu_seqlens=x["cu_seqlens"] if packed else None,
                           scale=d["scale"], out=out, final_state=fin, **kw)
    K.check_device_error()
    return o, f


def run_oracle(d, out_tokens=None):
    import oracle
    return oracle.recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"],
                            initial_state=d["initial_state"], cu_seqlens=d["cu_seqlens"],
                            scale=d["scale"], out_tokens=out_tokens)


def errs(x, ref):
    x = x.detach().double().cpu().numpy()
    assert np.isfinite(x).all(), "non-finite values (an output element was not written?)"
    rel = np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300)
    mx = np.max(np.abs(x - ref)) / max(np.max(np.abs(ref)), 1e-300)
    return rel, mx


def assert_parity(o, f, o_ref, f_ref, tag=""):
    for name, x, r in (("o", o, o_ref), ("final_state", f, f_ref)):
        rel, mx = errs(x, r)
        assert rel <= REL_L2 and mx <= MAX_ABS, f"{tag} {name}: rel_l2={rel:.3e} max={mx:.3e}"


# ------------------------------------------------ the five workloads

@pytest.mark.parametrize("name", ["tiny_T64_H1", "fixed_T8192_H64", "fixed_T8192_H96",
                                  "varlen16_T8192_H64"])
def test_workload_parity(name):
    d = KI.make_inputs(KI.WORKLOADS[name])
    o, f = run_gpu(d, packed=KI.WORKLOADS[name].varlen)
    o_ref, f_ref = run_oracle(d)
    assert_parity(o, f, o_ref, f_ref, name)


def test_long_context_parity():
    """T=131072, H=32: o on the first 8192 tokens, final state after all of them."""
    d = KI.make_inputs(KI.WORKLOADS["long_T131072_H32"])
    o, f = run_gpu(d, packed=False)
    o_ref, f_ref = run_oracle(d, out_tokens=8192)
    assert_parity(o[:8192], f, o_ref, f_ref, "long")


# ------------------------------------------------ ragged and degenerate

@pytest.mark.parametrize("T", [1, 2, 15, 16, 17, 31, 33, 100])
@pytest.mark.parametrize("init", [False, True])
def test_single_sequence_lengths(T, init):
    d = KI.make_case([T], H=2, seed=100 + T, init_state=init)
    o, f = run_gpu(d, packed=False)
    assert_parity(o, f, *run_oracle(d), f"T={T}")


def test_varlen_ragged_with_empty_sequences():
    d = KI.make_case([1, 0, 15, 16, 17, 100, 3, 0], H=3, seed=7, init_state=True)
    o, f = run_gpu(d, packed=True)
    assert_parity(o, f, *run_oracle(d), "ragged")


def test_fixed_batch_of_sequences():
    """B sequences of T tokens without cu_seqlens ([B, T, H, K] layout)."""
    Bn, T, H = 3, 37, 2
    d = KI.make_case([T] * Bn, H=H, seed=8, init_state=True)
    x = to_dev(d)
    q, k, v, g = (x[n].view(Bn, T, H, 128) for n in ("q", "k", "v", "g"))
    beta = x["beta"].view(Bn, T, H)
    o, f = K.chunk_prefill(q, k, v, g, beta, initial_state=x["initial_state"], scale=d["scale"])
    K.check_device_error()
    assert_parity(o.view(Bn * T, H, 128), f, *run_oracle(d), "batch")


def test_zero_tokens_copies_state():
    d = KI.make_case([0, 0], H=2, seed=9, init_state=True)
    x = to_dev(d)
    o, f = K.chunk_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"],
                           initial_state=x["initial_state"], cu_seqlens=x["cu_seqlens"])
    K.check_device_error()
    assert torch.equal(f, x["initial_state"])


def test_packed_equals_separate_calls_bitwise():
    d = KI.make_case([40, 7, 64, 19], H=2, seed=10, init_state=True)
    o, f = run_gpu(d, packed=True)
    cu = d["cu_seqlens"].tolist()
    for i in range(len(cu) - 1):
        a, b = cu[i], cu[i + 1]
        di = dict(q=d["q"][a:b], k=d["k"][a:b], v=d["v"][a:b], g=d["g"][a:b],
                  beta=d["beta"][a:b], initial_state=d["initial_state"][i:i + 1],
                  cu_seqlens=torch.tensor([0, b - a], dtype=torch.int32), seqlens=[b - a],
                  scale=d["scale"])
        oi, fi = run_gpu(di, packed=False)
        assert torch.equal(o[a:b], oi)
        assert torch.equal(f[i:i + 1], fi)


def test_split_call_equals_one_call():
    """State passing: prefill [0, T1) then [T1, T) from its final state."""
    d = KI.make_case([96], H=2, seed=11, init_state=True)
    o, f = run_gpu(d, packed=False)
    o_ref, f_ref = run_oracle(d)
    T1 = 48
    x = to_dev(d)
    s = slice(0, T1), slice(T1, 96)
    oa, fa = K.chunk_prefill(*(x[n][s[0]] for n in ("q", "k", "v", "g", "beta")),
                             initial_state=x["initial_state"], scale=d["scale"])
    ob, fb = K.chunk_prefill(*(x[n][s[1]].contiguous() for n in ("q", "k", "v", "g", "beta")),
                             initial_state=fa, scale=d["scale"])
    K.check_device_error()
    assert_parity(torch.cat([oa, ob]), fb, o_ref, f_ref, "split")
    # The second call starts from the first call's fp32 final state instead of
    # the state held inside the kernel (registers or tensor memory with its
    # lazily applied decay), so the two paths agree to rounding, not bitwise.
    rel_o, _ = errs(torch.cat([oa, ob]), o.double().cpu().numpy())
    rel_f, _ = errs(fb, f.double().cpu().numpy())
    assert rel_o <= 5e-3 and rel_f <= 5e-3, (rel_o, rel_f)


def test_in_place_state_and_no_final_state():
    d = KI.make_case([50], H=2, seed=12, init_state=True)
    o_ref, f_ref = run_oracle(d)
    x = to_dev(d)
    st = x["initial_state"].clone()
    o, f = K.chunk_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], initial_state=st,
                           final_state=st, scale=d["scale"])
    K.check_device_error()
    assert f.data_ptr() == st.data_ptr()
    assert_parity(o, st, o_ref, f_ref, "in-place")
    o2, f2 = K.chunk_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"],
                             initial_state=x["initial_state"], output_final_state=False,
                             scale=d["scale"])
    K.check_device_error()
    assert f2 is None and torch.equal(o2, o)


def test_segment_scan_strong_decay():
    """The exact form ahead of the segment-parallel scan (segment maps, their
    combine, then every segment at once), every other channel at -6 per token."""
    d = KI.make_case([1100], H=2, seed=46, init_state=True)
    d["g"][:, :, ::2] = -6.0
    o, f = run_gpu(d, packed=False)
    assert_parity(o, f, *run_oracle(d), "segment scan, strong decay")


@pytest.mark.parametrize("T,B,init", [(1024, 1, False), (2003, 1, True), (1040, 3, True),
                                      (4096, 2, False)])
def test_segment_scan_lengths(T, B, init):
    """Long fixed-length sequences with few heads take the segment-parallel
    scan on the 16-token path (here 4 to 16 segments, chosen from the SM
    count): odd chunk counts, a partial last chunk, several sequences."""
    H = 2
    d = KI.make_case([T] * B, H=H, seed=T + B, init_state=init)
    x = to_dev(d)
    q4 = {n: x[n].view(B, T, *x[n].shape[1:]) for n in ("q", "k", "v", "g", "beta")}
    o, f = K.chunk_prefill(q4["q"], q4["k"], q4["v"], q4["g"], q4["beta"],
                           initial_state=x["initial_state"], scale=d["scale"])
    K.check_device_error()
    o_ref, f_ref = run_oracle(d)
    assert_parity(o.view(B * T, H, 128), f, o_ref, f_ref)


def test_segment_scan_in_place_state():
    """An in-place state never takes the segment scan, and gives the same
    result as an out-of-place call."""
    T, H = 2048, 2
    d = KI.make_case([T], H=H, seed=8, init_state=True)
    x = to_dev(d)
    o1, f1 = K.chunk_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"],
                             initial_state=x["initial_state"], scale=d["scale"])
    st = x["initial_state"].clone()
    o2, f2 = K.chunk_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], initial_state=st,
                             scale=d["scale"], final_state=st)
    K.check_device_error()
    o_ref, f_ref = run_oracle(d)
    assert_parity(o2, st, o_ref, f_ref)
    assert_parity(o1, f1, o_ref, f_ref)


def scan_case(d, segments):
    """One fixed-length call with the segment count forced."""
    x = to_dev(d)
    B = len(d["seqlens"])
    T = d["seqlens"][0]
    q4 = {n: x[n].view(B, T, *x[n].shape[1:]) for n in ("q", "k", "v", "g", "beta")}
    try:
        assert K.kda_set_scan_segments(segments) == 0
        o, f = K.chunk_prefill(q4["q"], q4["k"], q4["v"], q4["g"], q4["beta"],
                               initial_state=x["initial_state"], scale=d["scale"])
        K.check_device_error()
    finally:
        K.kda_set_scan_segments(0)
    return o.view(B * T, *o.shape[2:]), f


@pytest.mark.parametrize("mu", [3.0, 7.0], ids=["decay", "weak_decay"])
@pytest.mark.parametrize("P", [2, 3, 8, 40])
def test_segment_scan_segments(P, mu, recurrent_impl):
    """P segments per sequence (segment maps built from the identity, the
    serial combine for P > 2, the replay): against the token recurrence and
    against the oracle's own segment-parallel form with P segments. 40
    segments of 3 or 4 chunks each on 126 chunks. With weak decay (log decay
    about -1e-3 per token) the entry states, hence the maps, carry over whole
    segments."""
    if recurrent_impl != 1:
        pytest.skip("the segment scan is on the 16-token path")
    import oracle
    d = KI.make_case([2003] * 2, H=2, seed=90 + P, init_state=True, mu=mu)
    o, f = scan_case(d, P)
    o_ref, f_ref = run_oracle(d)
    assert_parity(o, f, o_ref, f_ref, f"scan P={P}")
    o_s, f_s = oracle.segment_scan(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                   initial_state=d["initial_state"], cu_seqlens=d["cu_seqlens"],
                                   scale=d["scale"], segments=P)
    assert_parity(o, f, o_s, f_s, f"scan P={P} vs oracle segments")


def test_segment_scan_long_all_outputs(recurrent_impl):
    """T = 32768, H = 4, 8 segments of 256 chunks: every output token of
    every segment against the token recurrence, with a strongly decaying head
    (the exact form inside the segment maps) and a weakly decaying one."""
    if recurrent_impl != 1:
        pytest.skip("the segment scan is on the 16-token path")
    d = KI.make_case([32768], H=4, seed=97, init_state=True)
    d["g"][:, 3, ::3] = -6.0
    d["g"][:, 2, :] *= 0.02          # weak decay: the state carries across segments
    o, f = scan_case(d, 8)
    assert_parity(o, f, *run_oracle(d), "scan P=8 long")


def test_head_count_changes_between_calls():
    """7 heads, then 2, then 7 again on one stream (one workspace, never
    regrown): on the fused 64-token path the 2-head call puts its chunk
    offsets where the 7-head layout keeps ring counters, which the third call
    must find zeroed again."""
    for H, seqlens, seed in ((7, [150, 50], 120), (2, [100, 90], 121), (7, [150, 50], 122)):
        d = KI.make_case(seqlens, H=H, seed=seed, init_state=True)
        o, f = run_gpu(d)
        assert_parity(o, f, *run_oracle(d), f"H={H}")


def test_deterministic():
    d = KI.make_case([300], H=4, seed=13, init_state=True)
    o1, f1 = run_gpu(d, packed=False)
    o2, f2 = run_gpu(d, packed=False)
    assert torch.equal(o1, o2) and torch.equal(f1, f2)


def test_strong_decay_and_extreme_beta():
    """Decay just inside the factored range and beta at the ends of (0, 1)."""
    d = KI.make_case([64], H=2, seed=14, init_state=True)
    d["g"] = torch.full_like(d["g"], -4.5)          # 16 * 4.5 = 72 < 80 per chunk
    d["beta"][::2] = 1.0
    d["beta"][1::2] = 1e-4
    o, f = run_gpu(d, packed=False)
    assert_parity(o, f, *run_oracle(d), "strong-decay")


def test_scale_argument():
    d = KI.make_case([40], H=1, seed=15)
    d["scale"] = 0.37
    o, f = run_gpu(d, packed=False)
    assert_parity(o, f, *run_oracle(d), "scale")


# ------------------------------------------------ device-side errors

def test_bad_cu_seqlens_reported_and_outputs_untouched():
    d = KI.make_case([20, 30], H=1, seed=16)
    x = to_dev(d)
    bad = torch.tensor([0, 35, 30], dtype=torch.int32, device="cuda")  # decreasing, end != T
    out = torch.full_like(x["v"], 7.0)
    fin = torch.full((2, 1, 128, 128), 7.0, device="cuda")
    K.chunk_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], cu_seqlens=bad, out=out,
                    final_state=fin)
    rc = K.kda_last_device_error(torch.cuda.current_stream().cuda_stream)
    assert rc == K.STATUS_CODE["KDA_ERR_BAD_CU_SEQLENS"]
    assert bool((out == 7.0).all()) and bool((fin == 7.0).all())
    # the context is still usable and the flag was cleared
    o, f = run_gpu(d, packed=True)
    assert_parity(o, f, *run_oracle(d), "after-error")


def test_gate_growth_flagged():
    """Positive gates whose cumulative rise inside one chunk passes exp(80)
    have no finite form in fp32 (neither factored nor exact): the device
    flags them."""
    d = KI.make_case([32], H=1, seed=17)
    x = to_dev(d)
    x["g"].fill_(6.0)                                 # 16 * 6 = 96 > 80
    K.chunk_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"])
    rc = K.kda_last_device_error(torch.cuda.current_stream().cuda_stream)
    assert rc == K.STATUS_CODE["KDA_ERR_GATE_RANGE"]


def chunk_head_forms(d):
    """How many chunk-heads take each form of the gated products, by the
    intra-chunk kernel's rule on the cumulative log decay G of a chunk (nats,
    from 0 at the chunk start): factored about the chunk start when |G| <= 80
    everywhere; factored about the middle of G's range when that range
    (including the start) is at most 160 and G rises by at most 80; the exact
    per-pair form otherwise. The bounds are the kernel's, in base 2 (80 and
    160 nats with room for rounding: 115.42 and 230.84). Returns (start,
    middle, exact)."""
    log2e = 1.4426950408889634
    cu = d["cu_seqlens"].tolist()
    counts = [0, 0, 0]
    for n in range(len(cu) - 1):
        for t0 in range(cu[n], cu[n + 1], 16):
            G = d["g"][t0:min(t0 + 16, cu[n + 1])].double().cumsum(0)   # [L, H, 128]
            for h in range(G.shape[1]):
                g = G[:, h, :]
                if float(g.abs().max()) * log2e <= 115.42:
                    counts[0] += 1
                    continue
                hi, lo = max(0.0, float(g.max())), min(0.0, float(g.min()))
                low_so_far = torch.minimum(torch.cummin(g, 0).values, torch.zeros_like(g))
                before = torch.cat([torch.zeros_like(g[:1]), low_so_far[:-1]], 0)
                rise = float((g - before).max())
                counts[1 if ((hi - lo) * log2e <= 230.84 and rise * log2e <= 115.42) else 2] += 1
    return tuple(counts)


@pytest.mark.parametrize("gval", [-5.0, -5.001, -6.0, -10.0, -10.01, -60.0])
def test_strong_uniform_decay(gval):
    """The three forms of the gated products at their edges: -5 per token
    keeps |G| <= 80 (16 * 5 = 80) and factors about the chunk start; -5.001
    to -10 factor about the middle of the chunk's range (at most 160, which
    -10 reaches); -10.01 and -60 take the exact form. The 5-token tail chunk
    of the 37-token sequence stays in the first form. No flag."""
    d = KI.make_case([37, 16, 100], H=2, seed=31, init_state=True)
    d["g"] = torch.full_like(d["g"], gval)
    form = 0 if gval >= -5.0 else 1 if gval >= -10.0 else 2
    assert chunk_head_forms(d)[form] > 0
    o, f = run_gpu(d)
    assert_parity(o, f, *run_oracle(d), f"g={gval}")


def test_strong_mixed_decay_per_channel():
    """Per-channel decays from about 0 to below -20 per token (logsigmoid of
    N(-2, 4^2)), so chunks mix channels far outside the factored range with
    ordinary ones, in a ragged packed batch."""
    d = KI.make_case([200, 3, 77, 129], H=3, seed=32, init_state=True)
    gen = torch.Generator().manual_seed(33)
    x = torch.randn(d["g"].shape, generator=gen) * 4.0 - 2.0
    d["g"] = torch.nn.functional.logsigmoid(x)
    start, middle, exact = chunk_head_forms(d)
    assert start > 0 and middle > 0, (start, middle, exact)   # 54 and 30 of 84
    o, f = run_gpu(d)
    assert_parity(o, f, *run_oracle(d), "mixed")


def test_strong_decay_in_some_heads_only():
    """Two heads decay strongly, -9 per token (factored about the middle of
    the range) and -12 (exact form), the others not (factored about the
    chunk start): the three forms side by side in one launch."""
    d = KI.make_case([300], H=4, seed=34, init_state=True)
    d["g"][:, 2, :] = -9.0
    d["g"][:, 3, :] = -12.0
    assert all(n > 0 for n in chunk_head_forms(d))
    o, f = run_gpu(d)
    assert_parity(o, f, *run_oracle(d), "head 2 strong")


def test_host_pointer_rejected():
    d = KI.make_case([16], H=1, seed=18)
    x = to_dev(d)
    host_q = torch.zeros_like(d["q"])
    rc = K.kda_chunk_prefill(host_q.data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(),
                             x["g"].data_ptr(), x["beta"].data_ptr(), 0, 0, 1, 16, 1, 128, 128, 1,
                             1.0, torch.empty_like(x["v"]).data_ptr(), 0, 0)
    assert rc == K.STATUS_CODE["KDA_ERR_NOT_DEVICE_MEMORY"]


def test_graph_capture_after_warm_call():
    d = KI.make_case([128], H=2, seed=19, init_state=True)
    x = to_dev(d)
    out = torch.empty_like(x["v"])
    fin = torch.empty((1, 2, 128, 128), device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        K.chunk_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"],
                        initial_state=x["initial_state"], out=out, final_state=fin)
        s.synchronize()
        graph = torch.cuda.CUDAGraph()
        out.zero_()
        with torch.cuda.graph(graph, stream=s):
            K.chunk_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"],
                            initial_state=x["initial_state"], out=out, final_state=fin)
        graph.replay()
        s.synchronize()
    K.check_device_error()
    assert_parity(out, fin, *run_oracle(d), "graph")
