"""Pins of the fp64 oracle against facts fixed outside the oracle itself:
hand-worked examples, closed forms, special cases, library routines, an
independent product form of the recurrence, and brute force on tiny inputs.
CPU only."""

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), 'golden')
rng = np.random.default_rng(1234)


def _rand_unit(shape):
    x = rng.standard_normal(shape)
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


# ---------------------------------------------------------------- elementwise

def test_elementwise_closed_forms():
    assert O.sigmoid(0.0) == 0.5
    assert abs(O.softplus(0.0) - math.log(2.0)) < 1e-15
    assert O.silu(0.0) == 0.0
    x = np.linspace(-30, 30, 121)
    np.testing.assert_allclose(O.sigmoid(x) + O.sigmoid(-x), 1.0, atol=1e-15)
    np.testing.assert_allclose(O.softplus(x) - O.softplus(-x), x, atol=1e-12)
    ref = np.array([math.log1p(math.exp(t)) for t in x])
    np.testing.assert_allclose(O.softplus(x), ref, rtol=1e-14)
    ref_sig = np.array([1.0 / (1.0 + math.exp(-t)) for t in x])
    np.testing.assert_allclose(O.sigmoid(x), ref_sig, rtol=1e-14)
    np.testing.assert_allclose(O.silu(x), x * ref_sig, rtol=1e-14, atol=1e-300)
    assert np.isfinite(O.softplus(1e4)) and np.isfinite(O.sigmoid(-1e4))


def test_gating_closed_forms():
    Nv = 3
    a = np.zeros((2, Nv))
    b = np.zeros((2, Nv))
    A_log = np.array([0.0, math.log(3.0), math.log(0.5)])
    dt = np.zeros(Nv)
    g, beta = O.gating(a, b, A_log, dt)
    np.testing.assert_allclose(beta, 0.5)
    np.testing.assert_allclose(g[0], [-math.log(2), -3 * math.log(2), -0.5 * math.log(2)], rtol=1e-14)
    # a + dt_bias = 0 regardless of split
    g2, _ = O.gating(a + 0.7, b, A_log, dt - 0.7)
    np.testing.assert_allclose(g2, g, rtol=1e-14)
    # large positive pre-activation: softplus(x) ~ x, g ~ -exp(A_log) x
    g3, beta3 = O.gating(np.full((1, Nv), 40.0), np.full((1, Nv), 40.0), A_log, dt)
    np.testing.assert_allclose(g3[0], -np.exp(A_log) * 40.0, rtol=1e-15)
    assert np.all(beta3 <= 1.0) and np.all(g3 < 0)


# ----------------------------------------------------------------------- conv

def test_conv_hand_example():
    d = json.load(open(os.path.join(GOLDEN, 'conv_hand.json')))
    w = np.array(d['w'])[None, :]
    st = np.array(d['state'])[None, :]
    x = np.array(d['x'])[:, None]
    out, ns = O.causal_conv1d(x, w, None, st)
    np.testing.assert_array_equal(out[:, 0], d['out_pre_activation'])
    np.testing.assert_array_equal(ns[0], d['new_state'])


def test_conv_impulse_reproduces_taps():
    C, L, t0 = 5, 12, 4
    w = rng.standard_normal((C, 4))
    x = np.zeros((L, C))
    x[t0] = 1.0
    out, _ = O.causal_conv1d(x, w)
    for c in range(C):
        expect = np.zeros(L)
        for m in range(4):                    # w[c, 3] multiplies the current token
            expect[t0 + m] = w[c, 3 - m]
        np.testing.assert_array_equal(out[:, c], expect)


def test_conv_matches_numpy_convolve_and_bias():
    C, L = 7, 40
    w = rng.standard_normal((C, 4))
    bias = rng.standard_normal(C)
    x = rng.standard_normal((L, C))
    out, _ = O.causal_conv1d(x, w, bias)
    for c in range(C):
        ref = np.convolve(x[:, c], w[c, ::-1])[:L] + bias[c]
        np.testing.assert_allclose(out[:, c], ref, rtol=1e-13, atol=1e-13)


def test_conv_causality_and_state_carry():
    C, L = 6, 30
    w = rng.standard_normal((C, 4))
    x = rng.standard_normal((L, C))
    st = rng.standard_normal((C, 3))
    out, ns = O.causal_conv1d(x, w, None, st)
    x2 = x.copy()
    x2[17:] += 5.0
    out2, _ = O.causal_conv1d(x2, w, None, st)
    np.testing.assert_array_equal(out[:17], out2[:17])
    for cut in (1, 2, 3, 11):
        oa, sa = O.causal_conv1d(x[:cut], w, None, st)
        ob, sb = O.causal_conv1d(x[cut:], w, None, sa)
        np.testing.assert_allclose(np.concatenate([oa, ob]), out, rtol=1e-13, atol=1e-13)
        np.testing.assert_array_equal(sb, ns)
    np.testing.assert_array_equal(ns, x[-3:].T)
    # shorter than the window: the new state keeps part of the old one
    _, s1 = O.causal_conv1d(x[:1], w, None, st)
    np.testing.assert_array_equal(s1, np.concatenate([st[:, 1:], x[:1].T], axis=1))
    # no state == zero state
    o0, _ = O.causal_conv1d(x, w, None, None)
    oz, _ = O.causal_conv1d(x, w, None, np.zeros((C, 3)))
    np.testing.assert_array_equal(o0, oz)


# ---------------------------------------------------------------- norms

def test_l2norm_properties():
    x = rng.standard_normal((10, 3, 64)) * 5
    y = O.l2norm(x, 0.0)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(O.l2norm(3.5 * x, 0.0), y, rtol=1e-13)
    y_eps = O.l2norm(np.array([[3.0, 4.0]]), 11.0)          # sqrt(25 + 11) = 6
    np.testing.assert_allclose(y_eps, [[0.5, 4.0 / 6.0]], rtol=1e-15)


def test_gated_rmsnorm_properties():
    D = 16
    w = rng.standard_normal(D)
    z = rng.standard_normal((4, D))
    for c in (-2.5, 0.3, 7.0):
        y = O.gated_rmsnorm(np.full((4, D), c), z, w, eps=0.0)
        np.testing.assert_allclose(y, np.sign(c) * w * z / (1 + np.exp(-z)), rtol=1e-13)
    x = rng.standard_normal((4, D))
    np.testing.assert_array_equal(O.gated_rmsnorm(x, np.zeros((4, D)), w), 0.0)
    np.testing.assert_allclose(O.gated_rmsnorm(9.0 * x, z, w, eps=0.0),
                               O.gated_rmsnorm(x, z, w, eps=0.0), rtol=1e-13)
    # [3, 4]: mean square 12.5 (+ eps 0.5) -> rms sqrt(13)
    y = O.gated_rmsnorm(np.array([3.0, 4.0]), np.array([50.0, 50.0]), np.ones(2), eps=0.5)
    np.testing.assert_allclose(y, np.array([3.0, 4.0]) / math.sqrt(13.0) * 50.0, rtol=1e-14)


# ---------------------------------------------------------------- recurrence

def test_recurrence_hand_example():
    d = json.load(open(os.path.join(GOLDEN, 'delta_rule_hand.json')))
    q = np.array(d['q'])[:, None, :]
    k = np.array(d['k'])[:, None, :]
    v = np.array(d['v'])[:, None, :]
    g = np.array(d['g'])[:, None]
    beta = np.array(d['beta'])[:, None]
    o, S = O.recurrent_gated_delta_rule(q, k, v, g, beta)
    np.testing.assert_allclose(o[:, 0], d['o'], rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(S[0, 0], d['final_state'], rtol=1e-14, atol=1e-14)
    oc, Sc = O.chunk_gated_delta_rule(q, k, v, g, beta)
    np.testing.assert_allclose(oc[:, 0], d['o'], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(Sc[0, 0], d['final_state'], rtol=1e-13, atol=1e-13)


def test_recurrence_identity_when_gates_off():
    T, Nk, Nv, Dk, Dv = 9, 1, 2, 5, 3
    q = rng.standard_normal((T, Nk, Dk))
    k = rng.standard_normal((T, Nk, Dk))
    v = rng.standard_normal((T, Nv, Dv))
    S0 = rng.standard_normal((1, Nv, Dk, Dv))
    o, S = O.recurrent_gated_delta_rule(q, k, v, np.zeros((T, Nv)), np.zeros((T, Nv)),
                                        1.0, S0)
    np.testing.assert_array_equal(S, S0)
    for t in range(T):
        for h in range(Nv):
            for j in range(Dv):
                ref = sum(S0[0, h, i, j] * q[t, 0, i] for i in range(Dk))
                assert abs(o[t, h, j] - ref) < 1e-13


def test_recurrence_zero_key_pure_decay():
    T, Nv, Dk, Dv = 7, 2, 4, 6
    q = rng.standard_normal((T, 1, Dk))
    k = np.zeros((T, 1, Dk))
    v = rng.standard_normal((T, Nv, Dv))
    g = -rng.uniform(0, 2, (T, Nv))
    beta = rng.uniform(0, 1, (T, Nv))
    S0 = rng.standard_normal((1, Nv, Dk, Dv))
    o, S = O.recurrent_gated_delta_rule(q, k, v, g, beta, 1.0, S0)
    np.testing.assert_allclose(S[0], np.exp(g.sum(0))[:, None, None] * S0[0], rtol=1e-13)
    G = np.cumsum(g, 0)
    for t in range(T):
        ref = np.exp(G[t])[:, None] * np.einsum('hij,i->hj', S0[0], q[t, 0])
        np.testing.assert_allclose(o[t], ref, rtol=1e-12, atol=1e-14)
    # zero state stays zero
    _, Sz = O.recurrent_gated_delta_rule(q, k, v, g, beta)
    np.testing.assert_array_equal(Sz, 0.0)


def test_recurrence_unit_key_overwrites_row():
    Dk, Dv, Nv = 4, 3, 1
    S0 = rng.standard_normal((1, Nv, Dk, Dv))
    for i in range(Dk):
        k = np.zeros((1, 1, Dk))
        k[0, 0, i] = 1.0
        v = rng.standard_normal((1, Nv, Dv))
        q = rng.standard_normal((1, 1, Dk))
        _, S = O.recurrent_gated_delta_rule(q, k, v, np.zeros((1, Nv)), np.ones((1, Nv)), 1.0, S0)
        expect = S0[0, 0].copy()
        expect[i] = v[0, 0]
        np.testing.assert_allclose(S[0, 0], expect, rtol=1e-15, atol=1e-15)


def _product_form(q, k, v, g, beta, S0, scale):
    """S_t = (I - beta k k^T) exp(g) S_{t-1} + beta k v^T, o_t = S_t^T (scale q):
    the delta rule written as explicit matrix products, one head."""
    Dk = k.shape[1]
    S = S0.copy()
    outs = []
    for t in range(q.shape[0]):
        kk = np.outer(k[t], k[t])
        S = (np.eye(Dk) - beta[t] * kk) @ (math.exp(g[t]) * S) + beta[t] * np.outer(k[t], v[t])
        outs.append(S.T @ (scale * q[t]))
    return np.array(outs), S


def test_recurrence_matches_product_form_and_key_head_map():
    T, Nk, Nv, Dk, Dv = 11, 2, 4, 3, 2       # Dk != Dv catches a transposed state
    q = rng.standard_normal((T, Nk, Dk))
    k = _rand_unit((T, Nk, Dk))
    v = rng.standard_normal((T, Nv, Dv))
    g = -rng.uniform(0, 1.5, (T, Nv))
    beta = rng.uniform(0, 1, (T, Nv))
    S0 = rng.standard_normal((1, Nv, Dk, Dv))
    o, S = O.recurrent_gated_delta_rule(q, k, v, g, beta, 0.7, S0)
    for h in range(Nv):
        hk = h // (Nv // Nk)                 # repeat_interleave: 0,0,1,1
        ro, rS = _product_form(q[:, hk], k[:, hk], v[:, h], g[:, h], beta[:, h], S0[0, h], 0.7)
        np.testing.assert_allclose(o[:, h], ro, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(S[0, h], rS, rtol=1e-12, atol=1e-12)


def test_recurrence_exact_rational_brute_force():
    """Exact rational arithmetic of the product form on a 2x2 case vs the oracle."""
    F = Fraction
    k = [[F(3, 5), F(4, 5)], [F(1), F(0)], [F(0), F(1)]]
    v = [[F(1), F(2)], [F(-3), F(1, 2)], [F(2), F(-1)]]
    q = [[F(1), F(1)], [F(2), F(-1)], [F(1, 3), F(1)]]
    beta = [F(1, 2), F(1, 4), F(1)]
    alpha = [F(1), F(1, 2), F(1, 4)]
    S = [[F(0), F(0)], [F(0), F(0)]]
    outs = []
    for t in range(3):
        S = [[alpha[t] * S[i][j] for j in range(2)] for i in range(2)]
        Stk = [sum(S[i][j] * k[t][i] for i in range(2)) for j in range(2)]
        u = [beta[t] * (v[t][j] - Stk[j]) for j in range(2)]
        S = [[S[i][j] + k[t][i] * u[j] for j in range(2)] for i in range(2)]
        outs.append([sum(S[i][j] * q[t][i] for i in range(2)) for j in range(2)])
    f = lambda m: np.array(m, dtype=float)  # noqa: E731
    o, Sf = O.recurrent_gated_delta_rule(f(q)[:, None], f(k)[:, None], f(v)[:, None],
                                         np.log(f(alpha))[:, None], f(beta)[:, None])
    np.testing.assert_allclose(o[:, 0], f(outs), rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(Sf[0, 0], f(S), rtol=1e-14, atol=1e-15)


def test_recurrence_scale_is_linear():
    T, Dk, Dv = 5, 4, 4
    q = rng.standard_normal((T, 1, Dk))
    k = _rand_unit((T, 1, Dk))
    v = rng.standard_normal((T, 1, Dv))
    g = -rng.uniform(0, 1, (T, 1))
    beta = rng.uniform(0, 1, (T, 1))
    o1, S1 = O.recurrent_gated_delta_rule(q, k, v, g, beta, 1.0)
    o2, S2 = O.recurrent_gated_delta_rule(q, k, v, g, beta, 0.125)
    np.testing.assert_allclose(o2, 0.125 * o1, rtol=1e-14)
    np.testing.assert_array_equal(S1, S2)


# ---------------------------------------------------------------- chunked form

@pytest.mark.parametrize('lengths', [[1], [63], [64], [65], [200], [1, 64, 130, 7]])
def test_chunked_equals_recurrent(lengths):
    Nk, Nv, Dk, Dv = 2, 4, 16, 8
    T = sum(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)])
    q = _rand_unit((T, Nk, Dk))
    k = _rand_unit((T, Nk, Dk))
    v = rng.standard_normal((T, Nv, Dv))
    g = -np.exp(rng.uniform(0, math.log(16), Nv))[None] * O.softplus(rng.standard_normal((T, Nv)))
    beta = O.sigmoid(rng.standard_normal((T, Nv)))
    S0 = rng.standard_normal((len(lengths), Nv, Dk, Dv)) * 0.1
    o_r, S_r = O.recurrent_gated_delta_rule(q, k, v, g, beta, 0.25, S0, cu)
    o_c, S_c = O.chunk_gated_delta_rule(q, k, v, g, beta, 0.25, S0, cu)
    np.testing.assert_allclose(o_c, o_r, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(S_c, S_r, rtol=1e-9, atol=1e-11)
    o_16, S_16 = O.chunk_gated_delta_rule(q, k, v, g, beta, 0.25, S0, cu, chunk_size=16)
    np.testing.assert_allclose(o_16, o_r, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(S_16, S_r, rtol=1e-9, atol=1e-11)


def test_padding_tokens_are_identity():
    Nk, Nv, Dk, Dv, T, P = 1, 2, 8, 8, 70, 58
    q = _rand_unit((T, Nk, Dk))
    k = _rand_unit((T, Nk, Dk))
    v = rng.standard_normal((T, Nv, Dv))
    g = -rng.uniform(0, 3, (T, Nv))
    beta = rng.uniform(0, 1, (T, Nv))
    _, S = O.chunk_gated_delta_rule(q, k, v, g, beta)
    pad = lambda x: np.concatenate([x, np.zeros((P,) + x.shape[1:])])  # noqa: E731
    o_p, S_p = O.chunk_gated_delta_rule(pad(q), pad(k), pad(v), pad(g), pad(beta))
    np.testing.assert_allclose(S_p, S, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- end to end

def _mixer_case(T, B=1, seed=0, Nk=2, Nv=4, Dk=16, Dv=8):
    r = np.random.default_rng(seed)
    C = 2 * Nk * Dk + Nv * Dv
    return dict(
        mixed_qkv=r.standard_normal((T, C)), conv_w=r.standard_normal((C, 4)) * 0.5,
        a=r.standard_normal((T, Nv)), b=r.standard_normal((T, Nv)),
        A_log=r.uniform(0, math.log(16), Nv), dt_bias=r.uniform(-1, 1, Nv),
        z=r.standard_normal((T, Nv, Dv)), norm_w=1 + 0.1 * r.standard_normal(Dv),
        conv_state=r.standard_normal((B, C, 3)),
        S0=r.standard_normal((B, Nv, Dk, Dv)) * 0.1, dims=(Nk, Nv, Dk, Dv))


def test_decode_steps_equal_one_prefill():
    T = 9
    c = _mixer_case(T)
    Nk, Nv, Dk, Dv = c['dims']
    full = O.mixer_prefill(c['mixed_qkv'], c['conv_w'], c['a'], c['b'], c['A_log'], c['dt_bias'],
                           c['z'], c['norm_w'], Nk, Nv, Dk, Dv, conv_state=c['conv_state'],
                           initial_state=c['S0'])
    cs, S = c['conv_state'], c['S0']
    for t in range(T):
        d = O.decode_step(c['mixed_qkv'][t:t + 1], c['conv_w'], cs, c['a'][t:t + 1],
                          c['b'][t:t + 1], c['A_log'], c['dt_bias'], S, c['z'][t:t + 1],
                          c['norm_w'], Nk, Nv, Dk, Dv)
        np.testing.assert_allclose(d['y'][0], full['y'][t], rtol=1e-11, atol=1e-12)
        cs, S = d['conv_state'], d['state']
    np.testing.assert_allclose(S, full['state'], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(cs, full['conv_state'], rtol=0, atol=0)


def test_split_prefill_and_varlen_equal_whole():
    T = 150
    c = _mixer_case(T, B=1, seed=3)
    Nk, Nv, Dk, Dv = c['dims']
    args = lambda sl: (c['mixed_qkv'][sl], c['conv_w'], c['a'][sl], c['b'][sl], c['A_log'],  # noqa: E731
                       c['dt_bias'], c['z'][sl], c['norm_w'], Nk, Nv, Dk, Dv)
    full = O.mixer_prefill(*args(slice(0, T)), conv_state=c['conv_state'], initial_state=c['S0'],
                           use_chunked=True)
    p1 = O.mixer_prefill(*args(slice(0, 70)), conv_state=c['conv_state'], initial_state=c['S0'])
    p2 = O.mixer_prefill(*args(slice(70, T)), conv_state=p1['conv_state'],
                         initial_state=p1['state'])
    np.testing.assert_allclose(np.concatenate([p1['y'], p2['y']]), full['y'], rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(p2['state'], full['state'], rtol=1e-9, atol=1e-11)
    # packed varlen == separate calls
    lengths = [40, 1, 109]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    S0 = np.concatenate([c['S0']] * 3)
    cst = np.concatenate([c['conv_state']] * 3)
    packed = O.mixer_prefill(*args(slice(0, T)), cu_seqlens=cu, conv_state=cst, initial_state=S0)
    for s in range(3):
        sl = slice(cu[s], cu[s + 1])
        one = O.mixer_prefill(*args(sl), conv_state=c['conv_state'], initial_state=c['S0'])
        np.testing.assert_allclose(packed['y'][sl], one['y'], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(packed['state'][s], one['state'][0], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(packed['conv_state'][s], one['conv_state'][0], rtol=0, atol=0)


def test_conv_gating_split_and_scale():
    T = 12
    c = _mixer_case(T, seed=5)
    Nk, Nv, Dk, Dv = c['dims']
    cg = O.conv_gating(c['mixed_qkv'], c['conv_w'], c['a'], c['b'], c['A_log'], c['dt_bias'],
                       Nk, Nv, Dk, Dv, conv_state=c['conv_state'], l2_eps=0.0)
    np.testing.assert_allclose(np.linalg.norm(cg['q'], axis=-1), 1 / math.sqrt(Dk), rtol=1e-12)
    np.testing.assert_allclose(np.linalg.norm(cg['k'], axis=-1), 1.0, rtol=1e-12)
    # v is the silu of the conv of the last Nv*Dv channels, unnormalised
    out, _ = O.causal_conv1d(c['mixed_qkv'], c['conv_w'], None, c['conv_state'][0])
    np.testing.assert_allclose(cg['v'].reshape(T, -1), O.silu(out[:, 2 * Nk * Dk:]), rtol=1e-14)
    assert cg['g'].shape == (T, Nv) and np.all(cg['g'] < 0)


def _split_case():
    d = json.load(open(os.path.join(GOLDEN, 'qkv_split_hand.json')))
    dims = d['dims']
    x = np.array(d['x'])
    C = x.shape[1]
    w = np.zeros((C, 4))
    w[:, 3] = 1.0                                   # only the current token
    z = np.zeros((x.shape[0], dims['Nv']))
    return d, dims, x, w, z


def test_conv_gating_split_hand_example():
    # q = channels [0, Nk*Dk), k = the next Nk*Dk, v = the rest, each head-major
    d, dims, x, w, z = _split_case()
    cg = O.conv_gating(x, w, z, z, np.zeros(dims['Nv']), np.zeros(dims['Nv']), dims['Nk'], dims['Nv'],
                       dims['Dk'], dims['Dv'], q_scale=1 / math.sqrt(dims['Dk']), l2_eps=1e-6)
    np.testing.assert_allclose(cg['q'], d['q'], rtol=0, atol=1e-12)
    np.testing.assert_allclose(cg['k'], d['k'], rtol=0, atol=1e-12)
    np.testing.assert_allclose(cg['v'], d['v'], rtol=0, atol=1e-12)


def test_split_hand_example_tells_alternatives_apart():
    # the golden values differ from what a swapped [k | q] split or a (seq, head_dim, heads)
    # reshape would give, so either mistake in conv_gating fails the test above
    d, dims, x, w, z = _split_case()
    Nk, Dk, Nv, Dv = dims['Nk'], dims['Dk'], dims['Nv'], dims['Dv']
    y = O.silu(x)
    kd = Nk * Dk
    def norm(t):
        return O.l2norm(t, 1e-6)
    swapped_q = norm(y[:, kd:2 * kd].reshape(-1, Nk, Dk)) / math.sqrt(Dk)
    dim_major_q = norm(y[:, :kd].reshape(-1, Dk, Nk).transpose(0, 2, 1)) / math.sqrt(Dk)
    dim_major_v = y[:, 2 * kd:].reshape(-1, Dv, Nv).transpose(0, 2, 1)
    assert np.abs(swapped_q - np.array(d['q'])).max() > 0.1
    assert np.abs(dim_major_q - np.array(d['q'])).max() > 0.1
    assert np.abs(dim_major_v - np.array(d['v'])).max() > 0.1
