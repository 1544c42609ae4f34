"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test checks the oracle (both its recurrent and its chunked routine)
against something the pages or plain mathematics fix:
  * a hand-worked two-token example of the gated delta rule,
  * brute-force evaluation through explicit transition-matrix products,
  * closed forms (beta = 0, T = 1, orthonormal keys with beta = 1),
  * exact equality of the recurrent and chunk forms for several chunk sizes
    (the chunk form with C = 1 is the recurrence; C = L the parallel form),
  * split/resume, GVA head replication and sequence permutation invariants,
  * planted mistakes: an oracle with a dropped term or a wrong order fails,
  * the decode front-end: softplus and sigmoid at points with known values,
    the +-20 softplus branches against the exact function, alpha = 2^-c,
    the q/k norm as a sum of squares with eps inside the root, single-token
    closed forms, per-row length invariance, reduction to the plain step
    through independently inverted gates, and bf16 rounding against the
    library cast,
  * the output gate: silu at points with known values, the RMS of a constant
    row and of a one-hot row (a mean, not a sum), norm before gate, per-head
    normalisation,
  * the short convolution: the impulse response (weight orientation), the
    history feeding the first outputs, state of short and empty sequences,
    split/resume, slots and packed sequences, constant input.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_inputs(seed, lengths, hq, hv, dk, dv, s0=True, g_mu=0.0):
    rng = np.random.default_rng(seed)
    T = int(sum(lengths))
    unit = lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True)
    q = unit(rng.standard_normal((T, hq, dk)))
    k = unit(rng.standard_normal((T, hq, dk)))
    v = rng.standard_normal((T, hv, dv))
    g = -np.logaddexp(0, rng.standard_normal((T, hv)) + g_mu)
    beta = 1 / (1 + np.exp(-rng.standard_normal((T, hv))))
    S0 = 0.1 * rng.standard_normal((len(lengths), hv, dk, dv)) if s0 else None
    cu = np.concatenate([[0], np.cumsum(lengths)])
    return q, k, v, g, beta, S0, cu


def rel(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


# --------------------------------------------------------------------------
# hand-worked example (golden fixture, derivation in the file)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("routine", ["recurrent", "chunked1", "chunked2", "chunked64"])
def test_hand_example(routine):
    ex = json.load(open(os.path.join(GOLDEN, "hand_example_T2.json")))
    i = ex["inputs"]
    q = np.array(i["q"])[:, None, :]
    k = np.array(i["k"])[:, None, :]
    v = np.array(i["v"])[:, None, :]
    g = np.log(np.array(i["alpha"]))[:, None]
    beta = np.array(i["beta"])[:, None]
    cu = [0, 2]
    if routine == "recurrent":
        o, S = oracle.recurrent(q, k, v, g, beta, i["scale"], cu_seqlens=cu)
    else:
        o, S = oracle.chunked(q, k, v, g, beta, i["scale"], cu_seqlens=cu, chunk_size=int(routine[7:]))
    np.testing.assert_allclose(o[:, 0, :], ex["expected"]["o"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(S[0, 0], ex["expected"]["final_state"], rtol=0, atol=1e-14)


# --------------------------------------------------------------------------
# brute force through transition matrices, tiny sizes
#   S_t = T_t S_{t-1} + beta_t k_t^T v_t,  T_t = alpha_t (I - beta_t k_t^T k_t)
#   o_t = scale [q_t P_{t,0} S0 + sum_{i<=t} beta_i (q_t P_{t,i} k_i^T) v_i]
#   P_{t,i} = T_t ... T_{i+1}
# --------------------------------------------------------------------------
def brute_force(q, k, v, g, beta, scale, S0):
    T, dk = k.shape
    I = np.eye(dk)
    Tm = [np.exp(g[t]) * (I - beta[t] * np.outer(k[t], k[t])) for t in range(T)]
    o = np.zeros((T, v.shape[1]))
    scores = np.zeros((T, T))
    for t in range(T):
        P = I.copy()  # P_{t,t}
        for i in range(t, -1, -1):
            scores[t, i] = beta[i] * q[t] @ P @ k[i]
            P = P @ Tm[i]  # now P_{t,i-1}
        o[t] = scale * (q[t] @ P @ S0 + scores[t] @ v)
    # final state through the equivalent transition form of the update
    Sf = S0.copy()
    for t in range(T):
        Sf = Tm[t] @ Sf + beta[t] * np.outer(k[t], v[t])
    return o, Sf


@pytest.mark.parametrize("T,dk,dv,C", [(1, 4, 3, 64), (7, 4, 4, 3), (12, 8, 5, 4), (12, 6, 8, 64)])
def test_brute_force_tiny(T, dk, dv, C):
    q, k, v, g, beta, S0, cu = rand_inputs(7 + T, [T], 1, 1, dk, dv)
    o_bf, S_bf = brute_force(q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], 0.3, S0[0, 0])
    o_r, S_r = oracle.recurrent(q, k, v, g, beta, 0.3, S0, cu)
    o_c, S_c = oracle.chunked(q, k, v, g, beta, 0.3, S0, cu, chunk_size=C)
    for o, S in [(o_r, S_r), (o_c, S_c)]:
        assert rel(o[:, 0], o_bf) < 1e-12
        assert rel(S[0, 0], S_bf) < 1e-12


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------
@pytest.mark.parametrize("C", [1, 5, 64])
def test_beta_zero_pure_decay(C):
    """beta = 0: S_T = exp(sum g) S0 and o_t = scale exp(G_t) q_t S0."""
    q, k, v, g, beta, S0, cu = rand_inputs(3, [45], 2, 4, 8, 6)
    beta[:] = 0.0
    G = np.cumsum(g, axis=0)  # [T, Hv]
    hk = np.arange(4) // 2
    o_exp = 0.7 * np.exp(G)[:, :, None] * np.einsum("thd,hde->the", q[:, hk], S0[0])
    S_exp = np.exp(G[-1])[:, None, None] * S0[0]
    for o, S in [oracle.recurrent(q, k, v, g, beta, 0.7, S0, cu),
                 oracle.chunked(q, k, v, g, beta, 0.7, S0, cu, chunk_size=C)]:
        assert rel(o, o_exp) < 1e-12
        assert rel(S[0], S_exp) < 1e-12


def test_single_token_closed_form():
    """T = 1: S_1 = e^g S0 + beta k^T (v - e^g k S0), o = scale q S_1."""
    q, k, v, g, beta, S0, cu = rand_inputs(11, [1], 1, 2, 16, 16)
    for h in range(2):
        a = math.exp(g[0, h])
        S1 = a * S0[0, h] + beta[0, h] * np.outer(k[0, 0], v[0, h] - a * k[0, 0] @ S0[0, h])
        for o, S in [oracle.recurrent(q, k, v, g, beta, 0.5, S0, cu),
                     oracle.chunked(q, k, v, g, beta, 0.5, S0, cu)]:
            assert rel(S[0, h], S1) < 1e-13
            assert rel(o[0, h], 0.5 * q[0, 0] @ S1) < 1e-13


@pytest.mark.parametrize("with_s0", [False, True])
@pytest.mark.parametrize("C", [1, 4, 64])
def test_orthonormal_keys_overwrite(with_s0, C):
    """g = 0, beta = 1, orthonormal keys: each key reads back its own value.

    With beta = 1 and a unit key the old prediction is replaced by v exactly,
    and orthogonal keys do not disturb one another: k_j S_T = v_j for every j.
    Reading with q_t = k_j (j <= t) returns scale * v_j; with S0 = 0 a query
    orthogonal to all written keys reads zero.
    """
    rng = np.random.default_rng(5)
    dk, dv, T = 16, 8, 10
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    keys = Qm[:T]
    k = keys[:, None, :]
    v = rng.standard_normal((T, 1, dv))
    g = np.zeros((T, 1))
    beta = np.ones((T, 1))
    S0 = rng.standard_normal((1, 1, dk, dv)) if with_s0 else None
    js = rng.integers(0, np.arange(1, T + 1))  # j <= t
    q = keys[js][:, None, :]
    for o, S in [oracle.recurrent(q, k, v, g, beta, 0.5, S0, [0, T]),
                 oracle.chunked(q, k, v, g, beta, 0.5, S0, [0, T], chunk_size=C)]:
        np.testing.assert_allclose(keys @ S[0, 0], v[:, 0], atol=1e-12)
        np.testing.assert_allclose(o[:, 0], 0.5 * v[js, 0], atol=1e-12)
        if not with_s0:
            np.testing.assert_allclose(Qm[T:] @ S[0, 0], 0.0, atol=1e-12)


# --------------------------------------------------------------------------
# recurrent form == chunk form (the pages: C = 1 is the recurrence)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("C", [1, 7, 64, 200])
def test_chunked_equals_recurrent(C):
    q, k, v, g, beta, S0, cu = rand_inputs(21, [200], 2, 4, 32, 24)
    o_r, S_r = oracle.recurrent(q, k, v, g, beta, 0.125, S0, cu)
    o_c, S_c = oracle.chunked(q, k, v, g, beta, 0.125, S0, cu, chunk_size=C)
    assert rel(o_c, o_r) < 1e-11
    assert rel(S_c, S_r) < 1e-11


def test_chunked_equals_recurrent_varlen_full_dims():
    lengths = [0, 1, 63, 64, 65, 130]
    q, k, v, g, beta, S0, cu = rand_inputs(22, lengths, 1, 2, 128, 128)
    o_r, S_r = oracle.recurrent(q, k, v, g, beta, 1 / math.sqrt(128), S0, cu)
    o_c, S_c = oracle.chunked(q, k, v, g, beta, 1 / math.sqrt(128), S0, cu)
    assert rel(o_c, o_r) < 1e-11
    assert rel(S_c, S_r) < 1e-11
    # zero-length sequence: final state is the initial state
    np.testing.assert_array_equal(S_c[0], S0[0])


def test_dense_layout_matches_packed():
    q, k, v, g, beta, S0, cu = rand_inputs(23, [70, 70], 1, 1, 8, 8)
    o_p, S_p = oracle.chunked(q, k, v, g, beta, 1.0, S0, cu)
    shp = lambda x: x.reshape(2, 70, *x.shape[1:])
    o_d, S_d = oracle.chunked(shp(q), shp(k), shp(v), shp(g), shp(beta), 1.0, S0)
    np.testing.assert_array_equal(o_d.reshape(o_p.shape), o_p)
    np.testing.assert_array_equal(S_d, S_p)


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------
def test_split_resume():
    """Ch(T1) -> final -> Ch(T2, S0=final) equals Ch(T1+T2)."""
    q, k, v, g, beta, S0, cu = rand_inputs(31, [150], 1, 2, 16, 16)
    o_full, S_full = oracle.chunked(q, k, v, g, beta, 0.25, S0, cu)
    T1 = 71
    o_a, S_a = oracle.chunked(q[:T1], k[:T1], v[:T1], g[:T1], beta[:T1], 0.25, S0, [0, T1])
    o_b, S_b = oracle.chunked(q[T1:], k[T1:], v[T1:], g[T1:], beta[T1:], 0.25, S_a, [0, 150 - T1])
    assert rel(np.concatenate([o_a, o_b]), o_full) < 1e-12
    assert rel(S_b, S_full) < 1e-12


def test_gva_equals_replicated_heads():
    """Hv = G*Hq with shared q/k equals Hq = Hv with q/k heads repeated."""
    q, k, v, g, beta, S0, cu = rand_inputs(41, [90], 2, 6, 16, 8)
    o_g, S_g = oracle.chunked(q, k, v, g, beta, 0.3, S0, cu)
    rep = lambda x: np.repeat(x, 3, axis=1)
    o_r, S_r = oracle.chunked(rep(q), rep(k), v, g, beta, 0.3, S0, cu)
    np.testing.assert_array_equal(o_g, o_r)
    np.testing.assert_array_equal(S_g, S_r)


def test_sequence_permutation():
    """Reordering packed sequences reorders outputs bit for bit."""
    lengths = [33, 100, 7, 64]
    q, k, v, g, beta, S0, cu = rand_inputs(51, lengths, 1, 2, 16, 16)
    o, S = oracle.chunked(q, k, v, g, beta, 0.3, S0, cu)
    perm = [2, 0, 3, 1]
    segs = lambda x: [x[cu[i]:cu[i + 1]] for i in range(4)]
    cat = lambda x: np.concatenate([segs(x)[p] for p in perm])
    cu2 = np.concatenate([[0], np.cumsum([lengths[p] for p in perm])])
    o2, S2 = oracle.chunked(cat(q), cat(k), cat(v), cat(g), cat(beta), 0.3, S0[perm], cu2)
    np.testing.assert_array_equal(o2, cat(o))
    np.testing.assert_array_equal(S2, S[perm])


def test_recurrent_step_slots():
    """Decode wrapper: slot gather/scatter, negative index skips."""
    q, k, v, g, beta, _, _ = rand_inputs(61, [3], 1, 2, 8, 8)
    state = np.random.default_rng(1).standard_normal((5, 2, 8, 8))
    idx = np.array([4, -1, 1])
    o, st = oracle.recurrent_step(q, k, v, g, beta, 0.5, state, idx)
    o_ref, S_ref = oracle.recurrent(q[[0, 2]], k[[0, 2]], v[[0, 2]], g[[0, 2]], beta[[0, 2]], 0.5,
                                    state[[4, 1]], [0, 1, 2])
    np.testing.assert_array_equal(o[[0, 2]], o_ref)
    np.testing.assert_array_equal(o[1], 0.0)
    np.testing.assert_array_equal(st[[4, 1]], S_ref)
    np.testing.assert_array_equal(st[[0, 2, 3]], state[[0, 2, 3]])


# --------------------------------------------------------------------------
# planted mistakes (on the CPU, in a copy of the oracle's arithmetic) must be
# caught by the hand example: guards the pins themselves
# --------------------------------------------------------------------------
def _mutant_recurrent(q, k, v, alpha, beta, mode):
    S = np.zeros((k.shape[1], v.shape[1]))
    o = []
    for t in range(len(k)):
        if mode == "decay_after_write":
            S = S + beta[t] * np.outer(k[t], v[t] - k[t] @ S)
            S = alpha[t] * S
        elif mode == "read_before_write":
            S = alpha[t] * S
            o.append(q[t] @ S)
            S = S + beta[t] * np.outer(k[t], v[t] - k[t] @ S)
            continue
        elif mode == "no_prediction":
            S = alpha[t] * S + beta[t] * np.outer(k[t], v[t])
        o.append(q[t] @ S)
    return np.array(o), S


@pytest.mark.parametrize("mode", ["decay_after_write", "read_before_write", "no_prediction"])
def test_hand_example_catches_planted_mistakes(mode):
    ex = json.load(open(os.path.join(GOLDEN, "hand_example_T2.json")))
    i = ex["inputs"]
    o, S = _mutant_recurrent(np.array(i["q"]), np.array(i["k"]), np.array(i["v"]), i["alpha"], i["beta"], mode)
    bad = not (np.allclose(o, ex["expected"]["o"]) and np.allclose(S, ex["expected"]["final_state"]))
    assert bad


# --------------------------------------------------------------------------
# decode front-end (gates from the projections, q/k L2 norm): closed forms
# --------------------------------------------------------------------------
def test_softplus_closed_forms_and_branches():
    sp = oracle.softplus
    # interior: log(1 + e^x) at points where it is a known number
    np.testing.assert_allclose(sp(0.0), math.log(2.0), rtol=1e-15)
    np.testing.assert_allclose(sp(math.log(math.e - 1.0)), 1.0, rtol=1e-14)
    np.testing.assert_allclose(sp(math.log(math.exp(2.0) - 1.0)), 2.0, rtol=1e-14)
    x = np.linspace(-19.5, 19.5, 79)
    np.testing.assert_allclose(sp(x) - sp(-x), x, rtol=0, atol=1e-12)  # softplus(x) - softplus(-x) = x
    # the branches: identity above 20, e^x below -20, exactly
    assert sp(25.0) == 25.0 and sp(20.5) == 20.5
    assert sp(-25.0) == math.exp(-25.0) and sp(-20.5) == math.exp(-20.5)
    # and each branch is within e^-20 (relative) of the exact function
    for edge in (20.0, -20.0):
        xs = edge + np.linspace(-0.2, 0.2, 41)
        exact = np.logaddexp(0.0, xs)
        assert np.max(np.abs(sp(xs) - exact) / exact) < 2.1e-9


def test_decode_gates_closed_form():
    c = np.array([1.0, 2.0, 3.0, 0.5])
    A_log = np.log(c)
    # a + dt_bias = 0: softplus = ln 2, so g = -c ln 2 and alpha = 2^-c
    a = np.array([[1.3, -0.7, 0.0, 2.0]])
    dt_bias = -a[0]
    b = np.array([[0.0, math.log(3.0), -math.log(3.0), 40.0]])
    g, beta = oracle.decode_gates(a, b, A_log, dt_bias)
    np.testing.assert_allclose(np.exp(g), 2.0 ** -c[None], rtol=1e-14)
    np.testing.assert_allclose(beta, [[0.5, 0.75, 0.25, 1.0 / (1.0 + math.exp(-40.0))]], rtol=1e-15)
    # linear branch: a + dt_bias = 30 gives g = -30 c exactly
    g2, _ = oracle.decode_gates(np.full((1, 4), 31.0), b, A_log, np.full(4, -1.0))
    np.testing.assert_allclose(g2, -30.0 * c[None], rtol=1e-15)
    # sigmoid saturates without overflow warnings for large negative b
    _, b3 = oracle.decode_gates(a, np.full((1, 4), -800.0), A_log, dt_bias)
    assert np.all(b3 == 0.0)


def test_l2_normalise_is_sum_of_squares_with_eps_inside():
    x = np.zeros((2, 1, 128))
    x[0, 0, 0], x[0, 0, 1] = 3.0, 4.0
    y = oracle.l2_normalise(x)
    np.testing.assert_allclose(y[0, 0, :2], np.array([3.0, 4.0]) / math.sqrt(25.0 + 1e-6), rtol=1e-15)
    assert np.all(y[0, 0, 2:] == 0.0) and np.all(y[1] == 0.0)  # a zero row stays zero


def _gate_inputs_for(alpha_c, beta_b, hv):
    """a, b, A_log, dt_bias with alpha = 2^-alpha_c and beta = sigmoid(beta_b)."""
    A_log = np.log(np.full(hv, float(alpha_c)))
    return np.zeros((1, hv)), np.full((1, hv), float(beta_b)), A_log, np.zeros(hv)


@pytest.mark.parametrize("scale", [1.0 / math.sqrt(128.0), 0.37])
def test_gated_step_single_token_closed_form(scale):
    """S0 = 0, one token, q and k along e_0 with raw lengths 2 and 5:
    o = (q_bar . k_bar) beta v with q_bar . k_bar = scale * 2 * 5 / (sqrt(4 + eps) sqrt(25 + eps)),
    and the new state is k_bar^T (beta v): row 0 only."""
    dk = dv = 128
    hq, hv = 1, 2
    q = np.zeros((1, hq, dk)); q[0, 0, 0] = 2.0
    k = np.zeros((1, hq, dk)); k[0, 0, 0] = 5.0
    v = np.random.default_rng(3).standard_normal((1, hv, dv))
    a, _, A_log, dt_bias = _gate_inputs_for(1.0, 0.0, hv)
    b = np.array([[0.0, math.log(3.0)]])
    beta = np.array([0.5, 0.75])
    o, S = oracle.recurrent_step_gated(q, k, v, a, b, A_log, dt_bias, scale, np.zeros((1, hv, dk, dv)))
    qk = scale * 10.0 / (math.sqrt(4.0 + 1e-6) * math.sqrt(25.0 + 1e-6))
    np.testing.assert_allclose(o[0], qk * beta[:, None] * v[0], rtol=1e-13)
    np.testing.assert_allclose(S[0, :, 0, :], (5.0 / math.sqrt(25.0 + 1e-6)) * beta[:, None] * v[0], rtol=1e-13)
    assert np.all(S[0, :, 1:, :] == 0.0)


def test_gated_step_zero_key_only_decays():
    """k = 0 writes nothing: S' = 2^-c S0 and o = 2^-c q_bar S0 with q = 3 e_j."""
    dk = dv = 128
    hv, c, j, scale = 2, 3.0, 17, 0.25
    rng = np.random.default_rng(4)
    S0 = rng.standard_normal((1, hv, dk, dv))
    q = np.zeros((1, 1, dk)); q[0, 0, j] = 3.0
    a, b, A_log, dt_bias = _gate_inputs_for(c, 0.3, hv)
    o, S = oracle.recurrent_step_gated(q, np.zeros((1, 1, dk)), rng.standard_normal((1, hv, dv)),
                                       a, b, A_log, dt_bias, scale, S0)
    np.testing.assert_allclose(S, 2.0 ** -c * S0, rtol=1e-14)
    np.testing.assert_allclose(o[0], 2.0 ** -c * scale * 3.0 / math.sqrt(9.0 + 1e-6) * S0[0, :, j, :],
                               rtol=1e-13)


def test_gated_step_invariant_to_per_head_qk_lengths():
    """Normalisation is per (token, k-head) over d_k: rescaling each raw q/k
    row by its own factor (lengths far above sqrt(eps)) changes nothing."""
    rng = np.random.default_rng(5)
    N, hq, hv, dk, dv = 3, 2, 4, 16, 8
    q, k = rng.standard_normal((N, hq, dk)), rng.standard_normal((N, hq, dk))
    v = rng.standard_normal((N, hv, dv))
    a, b = rng.standard_normal((N, hv)), rng.standard_normal((N, hv))
    A_log, dt_bias = rng.uniform(0, 2, hv), rng.uniform(-4, 0, hv)
    S0 = rng.standard_normal((N, hv, dk, dv))
    o1, S1 = oracle.recurrent_step_gated(q, k, v, a, b, A_log, dt_bias, 0.3, S0)
    fq, fk = rng.uniform(1, 50, (N, hq, 1)), rng.uniform(1, 50, (N, hq, 1))
    o2, S2 = oracle.recurrent_step_gated(q * fq, k * fk, v, a, b, A_log, dt_bias, 0.3, S0)
    assert rel(o2, o1) < 1e-7 and rel(S2, S1) < 1e-7


def test_gated_step_reduces_to_plain_step():
    """Gates inverted independently (softplus^-1 through expm1, sigmoid^-1 as
    the logit) and keys of length 1000 (eps negligible) give back the plain
    decode step on the pre-normalised inputs."""
    rng = np.random.default_rng(6)
    N, hq, hv, dk, dv = 4, 2, 4, 32, 16
    q, k, v, g, beta, _, _ = rand_inputs(7, [N], hq, hv, dk, dv, s0=False)
    S0 = rng.standard_normal((N, hv, dk, dv))
    A_log = rng.uniform(-1, 2, hv)
    dt_bias = rng.uniform(-5, 1, hv)
    sp = -g / np.exp(A_log)[None]  # the softplus value each gate needs
    a = np.log(np.expm1(sp)) - dt_bias[None]
    b = np.log(beta / (1 - beta))
    o1, S1 = oracle.recurrent_step_gated(1000 * q, 1000 * k, v, a, b, A_log, dt_bias, 0.125, S0, [2, 0, 3, 1])
    o2, S2 = oracle.recurrent_step(q, k, v, g, beta, 0.125, S0, [2, 0, 3, 1])
    assert rel(o1, o2) < 1e-10 and rel(S1, S2) < 1e-10


def test_round_to_bf16_matches_library_cast():
    import torch

    rng = np.random.default_rng(8)
    x = np.concatenate([rng.uniform(0, 1, 4000), 10.0 ** rng.uniform(-45, 0, 2000),
                        # exact ties between two bf16 neighbours, both parities
                        (np.arange(256, 512) + 0.5) / 512.0, -rng.uniform(0, 3, 100), [0.0, 1.0]])
    lib = torch.tensor(x, dtype=torch.float64).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.round_to_bf16(x), lib)


def test_gated_step_beta_bf16_option():
    rng = np.random.default_rng(9)
    N, hq, hv, dk, dv = 2, 1, 2, 16, 8
    q, k = rng.standard_normal((N, hq, dk)), rng.standard_normal((N, hq, dk))
    v, a, b = rng.standard_normal((N, hv, dv)), rng.standard_normal((N, hv)), rng.standard_normal((N, hv))
    A_log, dt_bias, S0 = rng.uniform(0, 1, hv), rng.uniform(-3, 0, hv), rng.standard_normal((N, hv, dk, dv))
    o1, S1 = oracle.recurrent_step_gated(q, k, v, a, b, A_log, dt_bias, 0.5, S0, beta_bf16=True)
    g, beta = oracle.decode_gates(a, b, A_log, dt_bias)
    o2, S2 = oracle.recurrent_step(0.5 * oracle.l2_normalise(q), oracle.l2_normalise(k), v, g,
                                   oracle.round_to_bf16(beta), 1.0, S0)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(S1, S2)
    o3, _ = oracle.recurrent_step_gated(q, k, v, a, b, A_log, dt_bias, 0.5, S0)
    assert rel(o3, o1) > 1e-5  # the rounding is visible


# --------------------------------------------------------------------------
# output gate: head-wise RMSNorm, then SiLU(z)
# --------------------------------------------------------------------------
def test_silu_closed_forms():
    s = oracle.silu
    assert s(0.0)[0] == 0.0
    np.testing.assert_allclose(s(math.log(3.0)), 0.75 * math.log(3.0), rtol=1e-15)
    np.testing.assert_allclose(s(-math.log(3.0)), -0.25 * math.log(3.0), rtol=1e-15)
    x = np.linspace(-30, 30, 121)
    np.testing.assert_allclose(s(x) - s(-x), x, rtol=0, atol=1e-13)  # silu(x) - silu(-x) = x
    assert s(-800.0)[0] == 0.0 and s(800.0)[0] == 800.0


def test_gated_rmsnorm_constant_row():
    """o = c 1: the RMS is sqrt(c^2 + eps), so y = c / sqrt(c^2 + eps) w silu(z)."""
    rng = np.random.default_rng(11)
    d = 128
    w, z = rng.uniform(0.5, 2, d), rng.standard_normal((1, d))
    for c, eps in ((3.0, 1e-6), (-0.01, 1e-5), (2.0, 0.0)):
        y = oracle.gated_rmsnorm(np.full((1, d), c), z, w, eps)
        np.testing.assert_allclose(y, c / math.sqrt(c * c + eps) * w * oracle.silu(z), rtol=1e-14)


def test_gated_rmsnorm_mean_not_sum():
    """A single non-zero channel a: mean of squares a^2 / d, so y_0 = sqrt(d) w_0 silu(z_0) for eps = 0."""
    d = 128
    o = np.zeros((2, d)); o[0, 0] = 5.0; o[1, 7] = -0.25
    z = np.full((2, d), 1.5)
    w = np.linspace(0.5, 1.5, d)
    y = oracle.gated_rmsnorm(o, z, w, 0.0)
    g = 1.5 / (1.0 + math.exp(-1.5))
    np.testing.assert_allclose(y[0, 0], math.sqrt(d) * w[0] * g, rtol=1e-14)
    np.testing.assert_allclose(y[1, 7], -math.sqrt(d) * w[7] * g, rtol=1e-14)
    assert np.count_nonzero(y) == 2


def test_gated_rmsnorm_norm_before_gate_and_per_head():
    """The gate does not enter the RMS (y / silu(z) does not depend on z), and
    each head row is normalised on its own (rescaling one head leaves the
    others and, for eps = 0, itself unchanged)."""
    rng = np.random.default_rng(12)
    o = rng.standard_normal((3, 4, 128))
    w = rng.uniform(0.5, 2, 128)
    z1, z2 = rng.uniform(0.5, 3, o.shape), rng.uniform(-3, -0.5, o.shape)
    y1, y2 = oracle.gated_rmsnorm(o, z1, w, 1e-6), oracle.gated_rmsnorm(o, z2, w, 1e-6)
    np.testing.assert_allclose(y1 / oracle.silu(z1), y2 / oracle.silu(z2), rtol=1e-12)
    f = rng.uniform(0.1, 10, (3, 4, 1))
    np.testing.assert_allclose(oracle.gated_rmsnorm(o * f, z1, w, 0.0), oracle.gated_rmsnorm(o, z1, w, 0.0),
                               rtol=1e-12)


# --------------------------------------------------------------------------
# short causal convolution with its state
# --------------------------------------------------------------------------
def _silu1(v):
    return v / (1.0 + math.exp(-v))


def test_conv_impulse_response_fixes_orientation():
    """A unit impulse at t = 0 with zero history: the pre-activation at t is the
    weight of lag t, w[c, K-1-t] (oldest-first storage), then 0 after K taps."""
    w = np.array([[0.5, -1.0, 2.0, 3.0], [1.5, 0.25, -0.75, 1.0]])
    x = np.zeros((6, 2)); x[0] = [1.0, 2.0]
    out, st = oracle.causal_conv1d_silu(x, w, conv_state=np.zeros((1, 3, 2)))
    for t in range(6):
        for c in range(2):
            pre = x[0, c] * w[c, 3 - t] if t < 4 else 0.0
            np.testing.assert_allclose(out[t, c], _silu1(pre), rtol=1e-15, atol=1e-300)
    np.testing.assert_array_equal(st[0], x[3:])  # the last three inputs


def test_conv_history_feeds_the_first_outputs():
    """x = 0 with history [h0, h1, h2]: t = 0 sees w0 h0 + w1 h1 + w2 h2,
    t = 1 sees w0 h1 + w1 h2, t = 2 sees w0 h2, later outputs are silu(0) = 0;
    the bias adds to every pre-activation."""
    w = np.array([[2.0, -3.0, 0.5, 7.0]])
    h = np.array([[[1.0], [2.0], [-4.0]]])
    b = np.array([0.25])
    out, st = oracle.causal_conv1d_silu(np.zeros((5, 1)), w, b, h)
    pre = [2.0 * 1 - 3.0 * 2 + 0.5 * -4, 2.0 * 2 - 3.0 * -4, 2.0 * -4, 0.0, 0.0]
    np.testing.assert_allclose(out[:, 0], [_silu1(p + 0.25) for p in pre], rtol=1e-14)
    np.testing.assert_array_equal(st, np.zeros((1, 3, 1)))


def test_conv_short_sequences_keep_part_of_the_old_state():
    h = np.arange(6, dtype=float).reshape(1, 3, 2)
    w = np.ones((2, 4))
    x = np.array([[10.0, 20.0]])
    _, st1 = oracle.causal_conv1d_silu(x, w, conv_state=h)
    np.testing.assert_array_equal(st1[0], [[2, 3], [4, 5], [10, 20]])
    _, st0 = oracle.causal_conv1d_silu(np.zeros((0, 2)), w, conv_state=h, cu_seqlens=[0, 0])
    np.testing.assert_array_equal(st0, h)  # a zero-length sequence leaves its state


def test_conv_split_resume_and_slots():
    rng = np.random.default_rng(21)
    C, K = 8, 4
    w, b = rng.standard_normal((C, K)), rng.standard_normal(C)
    x = rng.standard_normal((50, C))
    h = rng.standard_normal((3, K - 1, C))
    full, st_full = oracle.causal_conv1d_silu(x, w, b, h, [0, 50], [2])
    a, st_a = oracle.causal_conv1d_silu(x[:17], w, b, h, [0, 17], [2])
    c, st_c = oracle.causal_conv1d_silu(x[17:], w, b, st_a, [0, 33], [2])
    np.testing.assert_allclose(np.concatenate([a, c]), full, rtol=1e-14)
    np.testing.assert_array_equal(st_c, st_full)
    np.testing.assert_array_equal(st_full[[0, 1]], h[[0, 1]])  # other slots untouched
    # packed sequences are independent; a negative slot means zero history and no write
    out2, st2 = oracle.causal_conv1d_silu(x[:30], w, b, h, [0, 12, 30], [-1, 1])
    o_a, _ = oracle.causal_conv1d_silu(x[:12], w, b, np.zeros((1, K - 1, C)))
    o_b, s_b = oracle.causal_conv1d_silu(x[12:30], w, b, h[[1]])
    np.testing.assert_allclose(out2, np.concatenate([o_a, o_b]), rtol=1e-14)
    np.testing.assert_array_equal(st2[1], s_b[0])
    np.testing.assert_array_equal(st2[[0, 2]], h[[0, 2]])


def test_conv_constant_input():
    """x = c everywhere, zero history: from t = K-1 on the window is full, so the
    pre-activation is c sum(w) + b."""
    w = np.array([[0.1, 0.2, 0.3, 0.4], [1.0, -1.0, 1.0, -1.0]])
    b = np.array([0.5, -0.5])
    out, _ = oracle.causal_conv1d_silu(np.full((7, 2), 3.0), w, b)
    np.testing.assert_allclose(out[3:, 0], _silu1(3.0 * 1.0 + 0.5), rtol=1e-14)
    np.testing.assert_allclose(out[3:, 1], _silu1(-0.5), rtol=1e-14)


def test_decode_precision_options():
    """bf16 beta and a bf16 state cache: the plain step on rounded beta, its
    updated slots rounded (both through the pinned bf16 rounding), other slots
    untouched."""
    q, k, v, g, beta, _, _ = rand_inputs(71, [3], 1, 2, 8, 8)
    state = oracle.round_to_bf16(np.random.default_rng(2).standard_normal((5, 2, 8, 8)))
    idx = np.array([4, -1, 1])
    o, st = oracle.recurrent_step(q, k, v, g, beta, 0.5, state, idx, beta_bf16=True, state_bf16=True)
    o2, st2 = oracle.recurrent_step(q, k, v, g, oracle.round_to_bf16(beta), 0.5, state, idx)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(st, oracle.round_to_bf16(st2))
    np.testing.assert_array_equal(st[[0, 2, 3]], state[[0, 2, 3]])
    assert np.all(oracle.round_to_bf16(st) == st)
