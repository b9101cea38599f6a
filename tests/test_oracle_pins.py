"""Pins of the fp64 oracle to facts other than itself.

Each check compares the oracle with something it does not compute the same
way: a closed form, a special case that reduces to textbook algebra, the
independently written chunked WY form, the explicit transition-matrix
products, hand-worked values, or an invariant of the recurrence. The
mutation test at the bottom plants each of a list of plausible mistakes in
the oracle and shows that at least one pin fails for it.
"""
import json
import os

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def _rand_case(rng, T, H, K, V, unit_k=True, s0=False, mu=3.0):
    f = np.float32
    q = rng.standard_normal((T, H, K)).astype(f)
    k = rng.standard_normal((T, H, K)).astype(f)
    if unit_k:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, V)).astype(f)
    x = rng.standard_normal((T, H, K)) + mu
    g = (-np.logaddexp(0.0, -x)).astype(f)         # logsigmoid
    beta = (1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))).astype(f)
    S0 = (0.5 * rng.standard_normal((1, H, K, V))) if s0 else None
    return q, k, v, g, beta, S0


def _relerr(a, b):
    d = np.max(np.abs(np.asarray(a) - np.asarray(b)))
    return d / max(np.max(np.abs(b)), 1e-300)


# ---------------------------------------------------------------- pins
# Each returns the error it measured; TOL holds the bound it must meet.

def pin_single_token(O, mutation=0):
    """T=1 from a zero state: o = scale beta (q.k) v and S = beta k v^T."""
    rng = np.random.default_rng(11)
    q, k, v, g, beta, _ = _rand_case(rng, 1, 3, 128, 128)
    o, S = O.recurrent(q, k, v, g, beta, mutation=mutation)
    sc = 1 / np.sqrt(128)
    qd, kd, vd, bd = (x.astype(np.float64) for x in (q, k, v, beta))
    o_ref = sc * bd[0, :, None] * np.einsum("hc,hc->h", qd[0], kd[0])[:, None] * vd[0]
    S_ref = bd[0, :, None, None] * np.einsum("hi,hj->hij", kd[0], vd[0])
    return max(_relerr(o[0], o_ref), _relerr(S[0], S_ref))


def pin_pure_decay(O, mutation=0):
    """beta=0: the state only decays, S_t = Diag(exp(sum_{u<=t} g_u)) S_0."""
    rng = np.random.default_rng(12)
    q, k, v, g, beta, S0 = _rand_case(rng, 40, 2, 128, 128, s0=True)
    beta[:] = 0.0
    o, S = O.recurrent(q, k, v, g, beta, initial_state=S0, mutation=mutation)
    G = np.cumsum(g.astype(np.float64), axis=0)              # [T, H, K]
    St = np.exp(G)[..., None] * S0[0][None]                  # [T, H, K, V]
    o_ref = (1 / np.sqrt(128)) * np.einsum("thij,thi->thj", St, q.astype(np.float64))
    return max(_relerr(o, o_ref), _relerr(S[0], St[-1]))


def pin_ungated_unrolled(O, mutation=0):
    """g=0 (ungated delta rule) against explicit transition-matrix products."""
    rng = np.random.default_rng(13)
    q, k, v, g, beta, S0 = _rand_case(rng, 4, 2, 16, 16, s0=True)
    g[:] = 0.0
    o, S = O.recurrent(q, k, v, g, beta, initial_state=S0, mutation=mutation)
    o_u, S_u = O.unrolled(q, k, v, g, beta, initial_state=S0[0])
    return max(_relerr(o, o_u), _relerr(S[0], S_u))


def pin_gated_unrolled(O, mutation=0, K=16, V=16):
    """General gates and betas against explicit transition-matrix products."""
    rng = np.random.default_rng(14)
    q, k, v, g, beta, S0 = _rand_case(rng, 4, 2, K, V, s0=True, mu=0.0)
    o, S = O.recurrent(q, k, v, g, beta, initial_state=S0, mutation=mutation)
    o_u, S_u = O.unrolled(q, k, v, g, beta, initial_state=S0[0])
    return max(_relerr(o, o_u), _relerr(S[0], S_u))


def pin_reset(O, mutation=0):
    """g -> -inf (exp(g) = 0 in fp64) erases the past: S_t = beta_t k_t v_t^T."""
    rng = np.random.default_rng(15)
    q, k, v, g, beta, S0 = _rand_case(rng, 6, 2, 128, 128, s0=True)
    g[:] = -1e4
    o, S = O.recurrent(q, k, v, g, beta, initial_state=S0, mutation=mutation)
    qd, kd, vd, bd = (x.astype(np.float64) for x in (q, k, v, beta))
    o_ref = (1 / np.sqrt(128)) * bd[..., None] * np.einsum("thc,thc->th", qd, kd)[..., None] * vd
    S_ref = bd[-1, :, None, None] * np.einsum("hi,hj->hij", kd[-1], vd[-1])
    return max(_relerr(o, o_ref), _relerr(S[0], S_ref))


def pin_exact_recall(O, mutation=0):
    """beta=1 and ||k||=1 exactly: (I - k k^T) is a projector, so k_t^T S_t = v_t^T."""
    rng = np.random.default_rng(16)
    T, H, K, V = 12, 2, 128, 128
    q, k, v, g, beta, S0 = _rand_case(rng, T, H, K, V, s0=True)
    k[:] = 0.0
    for t in range(T):
        for h in range(H):
            idx = rng.choice(K, 4, replace=False)
            k[t, h, idx] = 0.5 * rng.choice([-1.0, 1.0], 4)  # norm exactly 1 in binary
    beta[:] = 1.0
    worst = 0.0
    for t in range(1, T + 1):
        _, S = O.recurrent(q[:t], k[:t], v[:t], g[:t], beta[:t], initial_state=S0,
                           mutation=mutation)
        recall = np.einsum("hi,hij->hj", k[t - 1].astype(np.float64), S[0])
        worst = max(worst, _relerr(recall, v[t - 1].astype(np.float64)))
    return worst


def pin_chunked_form(O, mutation=0, Ts=(1, 15, 16, 17, 33, 64, 100), chunk=16):
    """The independently written chunk-wise WY form agrees with the recurrence."""
    rng = np.random.default_rng(17)
    worst = 0.0
    for T in Ts:
        q, k, v, g, beta, S0 = _rand_case(rng, T, 2, 128, 128, s0=True)
        o, S = O.recurrent(q, k, v, g, beta, initial_state=S0, mutation=mutation)
        oc, Sc = O.chunked(q, k, v, g, beta, initial_state=S0, chunk=chunk)
        worst = max(worst, _relerr(o, oc), _relerr(S, Sc))
    return worst


def pin_golden(O, mutation=0):
    """Hand-worked values (tests/golden/hand_worked_delta_rule.json)."""
    with open(os.path.join(HERE, "golden", "hand_worked_delta_rule.json")) as f:
        cases = json.load(f)["cases"]
    worst = 0.0
    for c in cases:
        q = np.array(c["q"], np.float32)[:, None, :]
        k = np.array(c["k"], np.float32)[:, None, :]
        v = np.array(c["v"], np.float32)[:, None, :]
        g = np.array(c["g"], np.float32)[:, None, :]
        beta = np.array(c["beta"], np.float32)[:, None]
        s0 = None if c["initial_state"] is None else np.array(c["initial_state"])[None, None]
        if mutation == 2 and c["K"] != c["V"]:
            continue
        o, S = O.recurrent(q, k, v, g, beta, initial_state=s0, scale=c["scale"],
                           mutation=mutation)
        err = max(np.max(np.abs(o[:, 0] - np.array(c["o"]))),
                  np.max(np.abs(S[0, 0] - np.array(c["final_state"]))))
        worst = max(worst, err / c["tol"] * 1e-12)  # normalised to the shared 1e-12 bound
    return worst


PINS = {
    "single_token": (pin_single_token, 1e-12),
    "pure_decay": (pin_pure_decay, 1e-10),
    "ungated_unrolled": (pin_ungated_unrolled, 1e-10),
    "gated_unrolled": (pin_gated_unrolled, 1e-10),
    "reset": (pin_reset, 1e-12),
    "exact_recall": (pin_exact_recall, 1e-12),
    "chunked_form": (pin_chunked_form, 1e-10),
    "golden": (pin_golden, 1e-12),
}


@pytest.mark.parametrize("name", list(PINS))
def test_pin(oracle_mod, name):
    fn, tol = PINS[name]
    assert fn(oracle_mod) <= tol


def test_unrolled_nonsquare(oracle_mod):
    assert pin_gated_unrolled(oracle_mod, K=8, V=12) <= 1e-10


@pytest.mark.parametrize("chunk", [1, 3, 7, 64])
def test_chunked_other_chunk_sizes(oracle_mod, chunk):
    assert pin_chunked_form(oracle_mod, Ts=(1, 17, 50), chunk=chunk) <= 1e-10


# ------------------------------------------------------------ invariants

def test_linearity_in_v_and_state(oracle_mod):
    """For fixed q, k, g, beta the map (V, S_0) -> (o, S_T) is linear."""
    O = oracle_mod
    rng = np.random.default_rng(21)
    q, k, _, g, beta, S1 = _rand_case(rng, 37, 2, 128, 128, s0=True)
    # values on a 2^-10 grid, so a*v1 + b*v2 below is exact in fp32
    v1 = (np.round(rng.standard_normal((37, 2, 128)) * 1024) / 1024).astype(np.float32)
    v2 = (np.round(rng.standard_normal((37, 2, 128)) * 1024) / 1024).astype(np.float32)
    S2 = rng.standard_normal(S1.shape)
    a, b = 1.0, -2.0
    o1, F1 = O.recurrent(q, k, v1, g, beta, initial_state=S1)
    o2, F2 = O.recurrent(q, k, v2, g, beta, initial_state=S2)
    vab = (a * v1 + b * v2).astype(np.float32)
    assert np.array_equal(vab.astype(np.float64), a * v1.astype(np.float64) + b * v2.astype(np.float64))
    oab, Fab = O.recurrent(q, k, vab, g, beta, initial_state=a * S1 + b * S2)
    assert _relerr(oab, a * o1 + b * o2) <= 1e-12
    assert _relerr(Fab, a * F1 + b * F2) <= 1e-12


def test_value_columns_separate(oracle_mod):
    """Permuting the value channels permutes o and the state's columns, exactly."""
    O = oracle_mod
    rng = np.random.default_rng(22)
    q, k, v, g, beta, S0 = _rand_case(rng, 29, 2, 128, 128, s0=True)
    perm = rng.permutation(128)
    o, F = O.recurrent(q, k, v, g, beta, initial_state=S0)
    op, Fp = O.recurrent(q, k, v[..., perm], g, beta, initial_state=S0[..., perm])
    assert np.array_equal(op, o[..., perm])
    assert np.array_equal(Fp, F[..., perm])


def test_state_passing(oracle_mod):
    """run(0:T) equals run(T1:T) started from run(0:T1)'s final state."""
    O = oracle_mod
    rng = np.random.default_rng(23)
    q, k, v, g, beta, S0 = _rand_case(rng, 53, 2, 128, 128, s0=True)
    o, F = O.recurrent(q, k, v, g, beta, initial_state=S0)
    for T1 in (1, 16, 21):
        oa, Fa = O.recurrent(q[:T1], k[:T1], v[:T1], g[:T1], beta[:T1], initial_state=S0)
        ob, Fb = O.recurrent(q[T1:], k[T1:], v[T1:], g[T1:], beta[T1:], initial_state=Fa)
        assert _relerr(np.concatenate([oa, ob]), o) <= 1e-12
        assert _relerr(Fb, F) <= 1e-12


def test_varlen_packed_equals_separate(oracle_mod):
    O = oracle_mod
    rng = np.random.default_rng(24)
    lens = [5, 0, 17, 32, 1]
    T = sum(lens)
    q, k, v, g, beta, _ = _rand_case(rng, T, 2, 128, 128)
    S0 = rng.standard_normal((len(lens), 2, 128, 128))
    cu = np.concatenate([[0], np.cumsum(lens)])
    for form in (O.recurrent, O.chunked):
        o, F = form(q, k, v, g, beta, initial_state=S0, cu_seqlens=cu)
        for i, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
            oi, Fi = form(q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b], initial_state=S0[i:i + 1])
            assert np.array_equal(o[a:b], oi)
            assert np.array_equal(F[i], Fi[0])


def test_empty_sequence_keeps_state(oracle_mod):
    O = oracle_mod
    rng = np.random.default_rng(25)
    q, k, v, g, beta, _ = _rand_case(rng, 3, 1, 128, 128)
    S0 = rng.standard_normal((2, 1, 128, 128))
    o, F = O.recurrent(q, k, v, g, beta, initial_state=S0, cu_seqlens=[0, 0, 3])
    assert np.array_equal(F[0], S0[0])


# ------------------------------------------------------------- mutations

MUTATIONS = {
    1: "output read from the pre-update state",
    2: "decay applied to value columns instead of key rows",
    3: "delta term added with the wrong sign",
    4: "beta dropped from the erase term",
    5: "decay applied after the delta update",
    6: "scale applied twice",
}


@pytest.mark.parametrize("m", list(MUTATIONS))
def test_each_planted_mistake_fails_a_pin(oracle_mod, m):
    failed = []
    for name, (fn, tol) in PINS.items():
        if name == "chunked_form":
            err = fn(oracle_mod, mutation=m, Ts=(17, 33))
        else:
            err = fn(oracle_mod, mutation=m)
        if not err <= tol:
            failed.append(name)
    assert failed, f"mutation {m} ({MUTATIONS[m]}) passed every pin"


# ---- input preprocessing (the kernels' flags): pinned against a library
# routine, a closed form and invariants, not against a retyped formula

def _raw_case(rng, T, H, K, V):
    q = rng.standard_normal((T, H, K)) * rng.uniform(0.25, 4.0, (T, H, 1))
    k = rng.standard_normal((T, H, K)) * rng.uniform(0.25, 4.0, (T, H, 1))
    v = rng.standard_normal((T, H, V))
    x = rng.standard_normal((T, H, K)) + 3.0
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    s0 = rng.standard_normal((1, H, K, V)) * 0.02
    f = lambda a: a.astype(np.float32)
    return f(q), f(k), f(v), f(x), f(beta), s0


def test_gate_logits_match_scipy_log_expit(oracle_mod):
    """logsigmoid of the logits inside the oracle == scipy.special.log_expit
    applied outside, including logits far out on both sides."""
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(5)
    q, k, v, x, beta, s0 = _raw_case(rng, 40, 2, 16, 8)
    x[3, 0, :4] = [30.0, -30.0, 0.0, 80.0]
    a = oracle_mod.recurrent(q, k, v, x, beta, s0, gate_logits=True, normalize_qk=True)
    g = special.log_expit(x.astype(np.float64)).astype(np.float32)
    b = oracle_mod.recurrent(q, k, v, g, beta, s0, normalize_qk=True)
    for u, w in zip(a, b):
        assert _relerr(u, w) < 1e-6


def test_gate_logit_zero_halves_the_state(oracle_mod):
    """beta = 0 and logit 0: logsigmoid(0) = -log 2, so every token halves S."""
    rng = np.random.default_rng(6)
    q, k, v, x, beta, s0 = _raw_case(rng, 9, 1, 8, 4)
    x[:] = 0.0
    beta[:] = 0.0
    _, fs = oracle_mod.recurrent(q, k, v, x, beta, s0, gate_logits=True)
    assert _relerr(fs, s0 * 0.5 ** 9) < 1e-12


def test_normalisation_is_scale_invariant(oracle_mod):
    """With normalize_qk, scaling any q or k row by a positive factor changes
    nothing (eps is negligible at these norms), and negating q flips o and
    leaves the state alone."""
    rng = np.random.default_rng(7)
    q, k, v, x, beta, s0 = _raw_case(rng, 30, 2, 16, 8)
    base = oracle_mod.recurrent(q, k, v, x, beta, s0, normalize_qk=True, gate_logits=True)
    c = rng.uniform(0.1, 10.0, (30, 2, 1)).astype(np.float32)
    scaled = oracle_mod.recurrent(q * c, k / c, v, x, beta, s0, normalize_qk=True,
                                  gate_logits=True)
    for u, w in zip(base, scaled):   # fp32 rounding of the scaled rows, carried over 30 tokens
        assert _relerr(u, w) < 1e-4
    o_neg, fs_neg = oracle_mod.recurrent(-q, k, v, x, beta, s0, normalize_qk=True,
                                         gate_logits=True)
    assert _relerr(o_neg, -base[0]) < 1e-12 and _relerr(fs_neg, base[1]) < 1e-12
    # without normalisation the same scaling does change the result
    plain = oracle_mod.recurrent(q, k, v, x, beta, s0, gate_logits=True)
    plain_s = oracle_mod.recurrent(q * c, k / c, v, x, beta, s0, gate_logits=True)
    assert _relerr(plain[1], plain_s[1]) > 1e-3


def test_normalisation_keeps_unit_rows(oracle_mod):
    """Rows that already have unit L2 norm pass through normalize_qk unchanged
    (up to eps and fp32 rounding of the inputs)."""
    rng = np.random.default_rng(8)
    q, k, v, x, beta, s0 = _raw_case(rng, 30, 2, 16, 8)
    qn = (q / np.linalg.norm(q.astype(np.float64), axis=-1, keepdims=True)).astype(np.float32)
    kn = (k / np.linalg.norm(k.astype(np.float64), axis=-1, keepdims=True)).astype(np.float32)
    a = oracle_mod.recurrent(qn, kn, v, x, beta, s0, normalize_qk=True, gate_logits=True)
    b = oracle_mod.recurrent(qn, kn, v, x, beta, s0, gate_logits=True)
    for u, w in zip(a, b):
        assert _relerr(u, w) < 2e-6
