"""Pins of the fp64 gradient oracle (oracle/kda_backward.c) against things
other than itself:

* its forward pass equals the forward oracle (kda_recurrent.c);
* every gradient equals central differences of that forward pass, along
  random directions, for each input separately;
* a single token from a zero state has closed-form gradients, written out
  here by hand;
* an empty sequence passes the final-state gradient straight through, and a
  packed batch equals its sequences run one by one;
* each planted mistake in the reverse pass fails a finite-difference pin;
* the chunk-wise reverse pass (oracle/chunked_backward.py), written from the
  chunk algebra, equals it at several chunk sizes.
"""
import numpy as np
import pytest
import torch

import kda_inputs as KI
import oracle


def case(seqlens, H=2, seed=0, init=True):
    d = KI.make_case(seqlens, H=H, seed=seed, init_state=init)
    gen = np.random.default_rng(seed + 100)
    T, N = sum(seqlens), len(seqlens)
    x = {n: d[n].double().numpy() for n in ("q", "k", "v", "g", "beta")}
    x["s0"] = None if d["initial_state"] is None else d["initial_state"].double().numpy()
    x["dout"] = gen.standard_normal((T, H, 128))
    x["dsf"] = gen.standard_normal((N, H, 128, 128)) * 0.1
    x["cu"] = d["cu_seqlens"].numpy().astype(np.int64)
    x["scale"] = d["scale"]
    return x


def run(x, **kw):
    return oracle.recurrent_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["dout"],
                                     initial_state=x["s0"], d_final_state=x["dsf"],
                                     cu_seqlens=x["cu"], scale=x["scale"], **kw)


def loss(x):
    r = run(x)
    return float(np.sum(r["o"] * x["dout"]) + np.sum(r["final_state"] * x["dsf"]))


GRAD = {"q": "dq", "k": "dk", "v": "dv", "g": "dg", "beta": "dbeta", "s0": "d_initial_state"}


def fd_error(x, name, grads, seed=1, eps=1e-6):
    """|central difference - <grad, direction>| / max(1, |<grad, direction>|)."""
    gen = np.random.default_rng(seed)
    dirn = gen.standard_normal(x[name].shape)
    xp, xm = dict(x), dict(x)
    xp[name] = x[name] + eps * dirn
    xm[name] = x[name] - eps * dirn
    fd = (loss(xp) - loss(xm)) / (2 * eps)
    an = float(np.sum(grads[GRAD[name]] * dirn))
    return abs(fd - an) / max(1.0, abs(an))


def test_forward_part_equals_forward_oracle():
    x = case([5, 0, 13], H=2, seed=3)
    r = run(x)
    o, fs = oracle.recurrent(torch.from_numpy(x["q"]).float(), torch.from_numpy(x["k"]).float(),
                             torch.from_numpy(x["v"]).float(), torch.from_numpy(x["g"]).float(),
                             torch.from_numpy(x["beta"]).float(), initial_state=x["s0"],
                             cu_seqlens=x["cu"], scale=x["scale"])
    np.testing.assert_allclose(r["o"], o, rtol=0, atol=1e-12 * np.abs(o).max())
    np.testing.assert_allclose(r["final_state"], fs, rtol=0, atol=1e-12 * np.abs(fs).max())


@pytest.mark.parametrize("name", list(GRAD))
def test_gradient_matches_central_differences(name):
    x = case([4, 7], H=2, seed=5)
    grads = run(x)
    for seed in (1, 2):
        assert fd_error(x, name, grads, seed=seed) < 1e-6, name


def test_gradients_with_strong_decay_and_no_initial_state():
    """Decays far outside the chunk kernels' factored range, and S_0 = 0."""
    x = case([9], H=1, seed=6, init=False)
    x["g"] = x["g"] * 0 - 7.0
    grads = run(x)
    for name in ("q", "k", "v", "g", "beta"):
        assert fd_error(x, name, grads) < 1e-6, name


def test_single_token_closed_form():
    """One token from S_0 = 0: S_1 = beta k v^T, o = scale beta (k.q) v, so
    L = scale beta (k.q)(v.dO) + beta k^T dSf v; its gradients by hand."""
    x = case([1], H=1, seed=7, init=False)
    r = run(x)
    q, k, v = x["q"][0, 0], x["k"][0, 0], x["v"][0, 0]
    dO, dSf, b, s = x["dout"][0, 0], x["dsf"][0, 0], x["beta"][0, 0], x["scale"]
    a = np.exp(x["g"][0, 0])
    kq, vd = k @ q, v @ dO
    np.testing.assert_allclose(r["dq"][0, 0], s * b * vd * k, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(r["dk"][0, 0], s * b * vd * q + b * dSf @ v, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(r["dv"][0, 0], s * b * kq * dO + b * dSf.T @ k, rtol=1e-12,
                               atol=1e-14)
    np.testing.assert_allclose(r["dbeta"][0, 0], s * kq * vd + k @ dSf @ v, rtol=1e-12)
    np.testing.assert_array_equal(r["dg"][0, 0], np.zeros(128))   # S_0 = 0
    # dL/dS_0: the state gradient (dSf + s q dO^T) with the erase term, times a
    dS = dSf + s * np.outer(q, dO)
    x_ = dS.T @ k
    ds0 = a[:, None] * (dS - b * np.outer(k, x_))
    np.testing.assert_allclose(r["d_initial_state"][0, 0], ds0, rtol=1e-12, atol=1e-14)


def test_empty_sequence_passes_state_gradient_through():
    x = case([6, 0, 3], H=2, seed=8)
    r = run(x)
    np.testing.assert_array_equal(r["d_initial_state"][1], x["dsf"][1])


def test_packed_equals_separate_sequences():
    x = case([5, 8], H=2, seed=9)
    r = run(x)
    for n, (a, b) in enumerate([(0, 5), (5, 13)]):
        y = dict(x)
        for key in ("q", "k", "v", "g", "beta", "dout"):
            y[key] = x[key][a:b]
        y["s0"], y["dsf"] = x["s0"][n:n + 1], x["dsf"][n:n + 1]
        y["cu"] = np.array([0, b - a], dtype=np.int64)
        ry = run(y)
        for key in ("dq", "dk", "dv", "dg", "dbeta"):
            np.testing.assert_array_equal(r[key][a:b], ry[key])
        np.testing.assert_array_equal(r["d_initial_state"][n], ry["d_initial_state"][0])


@pytest.mark.parametrize("mutation", [1, 2, 3, 4, 5])
def test_each_planted_mistake_fails_a_pin(mutation):
    x = case([4, 7], H=1, seed=10)
    grads = run(x, mutation=mutation)
    worst = max(fd_error(x, name, grads) for name in GRAD)
    assert worst > 1e-3, (mutation, worst)


def chunked(x, chunk):
    return oracle.chunked_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["dout"],
                                   initial_state=x["s0"], d_final_state=x["dsf"],
                                   cu_seqlens=x["cu"], scale=x["scale"], chunk=chunk)


KEYS = ("o", "final_state", "dq", "dk", "dv", "dg", "dbeta", "d_initial_state")


@pytest.mark.parametrize("chunk", [1, 3, 16, 64])
def test_chunked_reverse_pass_equals_token_reverse_pass(chunk):
    x = case([37, 0, 20, 16], H=2, seed=12)
    ref, got = run(x), chunked(x, chunk)
    for key in KEYS:
        np.testing.assert_allclose(got[key], ref[key], rtol=0,
                                   atol=1e-12 * max(1.0, np.abs(ref[key]).max()), err_msg=key)


def test_chunked_reverse_pass_strong_decay_no_states():
    """Per-pair exponentials of the chunk form at decays far past the
    factored range; no initial state and no final-state gradient."""
    x = case([40], H=1, seed=13, init=False)
    x["g"] = x["g"] * 0 - 8.0
    x["dsf"] = None
    ref, got = run(x), chunked(x, 16)
    for key in KEYS:
        np.testing.assert_allclose(got[key], ref[key], rtol=0,
                                   atol=1e-12 * max(1.0, np.abs(ref[key]).max()), err_msg=key)
