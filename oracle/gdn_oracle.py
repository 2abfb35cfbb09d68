"""Plain fp64 CPU oracle of the Gated DeltaNet token mixer.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` call it.  It shares no code with the CUDA library.

Every function is written from the plain definition of the step it computes,
in NumPy float64, token by token where the method is a recurrence.  Sources
(page title, section):

* "Qwen3.5 Dense Model Architecture", section "Linear Attention" -- the
  forward listing (causal conv with cached left context, split into q/k/v
  heads, beta = sigmoid(b), g = -exp(A_log) * softplus(a + dt_bias) in fp32,
  key heads repeated to the value-head count, recurrent or chunked delta
  rule with optional initial state and final state, gated RMSNorm with z),
  and section "Cache 组织" (conv_states [B, conv_dim, K],
  recurrent_states [B, Nv, Dk, Dv]).
* "Qwen3.5 Simulation Support Design Document", section 2.2 (the seven
  linear-attention ops: conv + SiLU, fused gating with the q/k L2-norm,
  chunk / recurrent delta rule, gated RMSNorm) and Appendix B (chunk size 64,
  intra-chunk attention plus inter-chunk recurrence).

Readings where the pages are silent (each is listed in the design doc):
conv state keeps the last K-1 = 3 raw inputs, oldest first; PyTorch
cross-correlation tap order (w[:, K-1] multiplies the current token); SiLU
after the conv on both paths; L2-norm x / sqrt(sum x^2 + eps); RMSNorm
x / sqrt(mean x^2 + eps) * w * silu(z) (plain weight, not 1 + weight);
q scaled by 1/sqrt(Dk) after its L2-norm; the output read is o_t = S_t^T q_t
with S laid out [Dk, Dv].

Array conventions (all token-major, sequences packed back to back):
  mixed_qkv [tokens, C], C = 2*Nk*Dk + Nv*Dv, split [q | k | v]
  q, k [tokens, Nk, Dk]; v [tokens, Nv, Dv]; a, b, g, beta [tokens, Nv]
  conv_w [C, K]; conv_state [N, C, K-1]; state [N, Nv, Dk, Dv]
  cu_seqlens [N+1] (int), cu_seqlens[0] = 0, non-decreasing.
"""

import numpy as np

CONV_K = 4          # kernel size of the depthwise causal conv
CHUNK = 64          # chunk length of the chunked delta rule


def _f64(x):
    return None if x is None else np.asarray(x, dtype=np.float64)


def _seq_bounds(cu_seqlens, total_tokens, num_seqs=1):
    """(bos, eos) of every packed sequence; equal split when cu_seqlens is None."""
    if cu_seqlens is None:
        assert total_tokens % num_seqs == 0
        L = total_tokens // num_seqs
        return [(s * L, (s + 1) * L) for s in range(num_seqs)]
    cu = [int(c) for c in np.asarray(cu_seqlens).reshape(-1)]
    return [(cu[i], cu[i + 1]) for i in range(len(cu) - 1)]


# ---------------------------------------------------------------------------
# elementwise functions
# ---------------------------------------------------------------------------

def sigmoid(x):
    """1 / (1 + e^-x), evaluated as exp(-log(1 + e^-x)) to stay finite."""
    x = _f64(x)
    return np.exp(-np.logaddexp(0.0, -x))


def softplus(x):
    """log(1 + e^x)."""
    return np.logaddexp(0.0, _f64(x))


def silu(x):
    """x * sigmoid(x)."""
    x = _f64(x)
    return x * sigmoid(x)


# ---------------------------------------------------------------------------
# a1: depthwise causal conv with state carry-over
# ---------------------------------------------------------------------------

def causal_conv1d(x, conv_w, conv_bias=None, conv_state=None):
    """Depthwise causal conv of one sequence, before the activation.

    Linear Attention listing: when a cached state exists it is concatenated in
    front of the new inputs along time, the conv runs over the result, and only
    the last seq_len outputs are kept; the cache keeps the tail of the raw
    (pre-conv) inputs.

    x [L, C]; conv_w [C, K]; conv_bias [C] or None; conv_state [C, K-1] or
    None (zeros).  Returns (out [L, C], new_state [C, K-1]).
    out[t, c] = bias[c] + sum_j w[c, j] * xpad[t + j, c], xpad = [state ; x].
    """
    x = _f64(x)
    w = _f64(conv_w)
    L, C = x.shape
    K = w.shape[1]
    state = np.zeros((C, K - 1)) if conv_state is None else _f64(conv_state)
    xpad = np.concatenate([state.T, x], axis=0)          # [K-1+L, C]
    out = np.zeros((L, C))
    for j in range(K):
        out += w[:, j][None, :] * xpad[j:j + L]
    if conv_bias is not None:
        out += _f64(conv_bias)[None, :]
    new_state = xpad[L:L + K - 1].T.copy()               # last K-1 raw inputs
    return out, new_state


def l2norm(x, eps):
    """x / sqrt(sum(x^2) + eps) over the last axis."""
    x = _f64(x)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def gating(a, b, A_log, dt_bias):
    """beta = sigmoid(b); g = -exp(A_log) * softplus(a + dt_bias).

    Linear Attention listing; g is the per-token, per-value-head log-decay.
    """
    beta = sigmoid(b)
    g = -np.exp(_f64(A_log))[None, :] * softplus(_f64(a) + _f64(dt_bias)[None, :])
    return g, beta


def conv_gating(mixed_qkv, conv_w, a, b, A_log, dt_bias, Nk, Nv, Dk, Dv,
                cu_seqlens=None, num_seqs=1, conv_bias=None, conv_state=None,
                q_scale=None, l2_eps=1e-6):
    """a1 + a2 + a3: conv + SiLU + split + L2-norm + q scale + gating.

    Returns dict q [T, Nk, Dk], k [T, Nk, Dk], v [T, Nv, Dv], g, beta [T, Nv],
    conv_state [N, C, K-1].
    """
    x = _f64(mixed_qkv)
    T, C = x.shape
    assert C == 2 * Nk * Dk + Nv * Dv
    if q_scale is None:
        q_scale = 1.0 / np.sqrt(Dk)
    bounds = _seq_bounds(cu_seqlens, T, num_seqs)
    y = np.zeros((T, C))
    states = np.zeros((len(bounds), C, CONV_K - 1))
    for s, (bos, eos) in enumerate(bounds):
        st = None if conv_state is None else conv_state[s]
        out, new_state = causal_conv1d(x[bos:eos], conv_w, conv_bias, st)
        y[bos:eos] = silu(out)
        states[s] = new_state
    kd = Nk * Dk
    q = y[:, :kd].reshape(T, Nk, Dk)
    k = y[:, kd:2 * kd].reshape(T, Nk, Dk)
    v = y[:, 2 * kd:].reshape(T, Nv, Dv)
    q = l2norm(q, l2_eps) * q_scale
    k = l2norm(k, l2_eps)
    g, beta = gating(a, b, A_log, dt_bias)
    return dict(q=q, k=k, v=v.copy(), g=g, beta=beta, conv_state=states)


# ---------------------------------------------------------------------------
# a5: the recurrent gated delta rule, token by token
# ---------------------------------------------------------------------------

def _value_to_key_head(Nk, Nv):
    """repeat_interleave of key heads: value head h reads key head h // (Nv/Nk)."""
    assert Nv % Nk == 0
    return np.arange(Nv) // (Nv // Nk)


def recurrent_gated_delta_rule(q, k, v, g, beta, scale=1.0, initial_state=None,
                               cu_seqlens=None, num_seqs=1):
    """Token-by-token gated delta rule.

    For each sequence and value head h (key head h // r), from S = S0 or 0:
        S   <- exp(g_t) * S
        u   =  beta_t * (v_t - S^T k_t)
        S   <- S + k_t u^T
        o_t =  S^T (scale * q_t)
    S is [Dk, Dv].  Returns (o [T, Nv, Dv], final_state [N, Nv, Dk, Dv]).
    """
    q, k, v, g, beta = (_f64(t) for t in (q, k, v, g, beta))
    T, Nk, Dk = q.shape
    Nv, Dv = v.shape[1], v.shape[2]
    hk = _value_to_key_head(Nk, Nv)
    bounds = _seq_bounds(cu_seqlens, T, num_seqs)
    o = np.zeros((T, Nv, Dv))
    finals = np.zeros((len(bounds), Nv, Dk, Dv))
    for s, (bos, eos) in enumerate(bounds):
        S = np.zeros((Nv, Dk, Dv)) if initial_state is None else _f64(initial_state[s]).copy()
        for t in range(bos, eos):
            qt = q[t, hk] * scale                       # [Nv, Dk]
            kt = k[t, hk]
            S *= np.exp(g[t])[:, None, None]
            u = beta[t][:, None] * (v[t] - np.einsum('hkv,hk->hv', S, kt))
            S += kt[:, :, None] * u[:, None, :]
            o[t] = np.einsum('hkv,hk->hv', S, qt)
        finals[s] = S
    return o, finals


# ---------------------------------------------------------------------------
# a4: the chunked form (fp64), used to check chunked == recurrent
# ---------------------------------------------------------------------------

def chunk_gated_delta_rule(q, k, v, g, beta, scale=1.0, initial_state=None,
                           cu_seqlens=None, num_seqs=1, chunk_size=CHUNK,
                           keep=None):
    """Chunked gated delta rule, chunks restart at every sequence start.

    Within a chunk of length L with entry state S0 and G = cumsum(g):
      A[r,j] = beta_r exp(G_r - G_j) k_r.k_j   (j < r)
      (I + A) [U~ | W] = [diag(beta) V | diag(beta exp(G)) K]
      U = U~ - W S0
      O = diag(exp(G)) Q S0 + (M o Q K^T) U,  M[r,j] = exp(G_r - G_j), j <= r
      S_L = exp(G_L) S0 + (diag(exp(G_L - G)) K)^T U
    This is the recurrence of recurrent_gated_delta_rule unrolled over the
    chunk (the u_t of the recurrence are the rows of U).  ``keep`` optionally
    restricts which token rows of o are stored (a boolean mask [T]) so that
    very long sequences need not hold every output.
    """
    q, k, v, g, beta = (_f64(t) for t in (q, k, v, g, beta))
    T, Nk, Dk = q.shape
    Nv, Dv = v.shape[1], v.shape[2]
    hk = _value_to_key_head(Nk, Nv)
    bounds = _seq_bounds(cu_seqlens, T, num_seqs)
    o = np.zeros((T, Nv, Dv))
    finals = np.zeros((len(bounds), Nv, Dk, Dv))
    for s, (bos, eos) in enumerate(bounds):
        S = np.zeros((Nv, Dk, Dv)) if initial_state is None else _f64(initial_state[s]).copy()
        for c0 in range(bos, eos, chunk_size):
            c1 = min(c0 + chunk_size, eos)
            L = c1 - c0
            Qc = np.transpose(q[c0:c1][:, hk], (1, 0, 2)) * scale    # [Nv, L, Dk]
            Kc = np.transpose(k[c0:c1][:, hk], (1, 0, 2))
            Vc = np.transpose(v[c0:c1], (1, 0, 2))                   # [Nv, L, Dv]
            bc = beta[c0:c1].T                                       # [Nv, L]
            G = np.cumsum(g[c0:c1].T, axis=1)                        # [Nv, L]
            diff = G[:, :, None] - G[:, None, :]                     # G_r - G_j
            lower = np.tril(np.ones((L, L), dtype=bool), -1)
            lower_eq = np.tril(np.ones((L, L), dtype=bool), 0)
            dec_strict = np.exp(np.where(lower, diff, -np.inf))
            dec = np.exp(np.where(lower_eq, diff, -np.inf))
            KK = Kc @ np.transpose(Kc, (0, 2, 1))
            A = bc[:, :, None] * dec_strict * KK
            I = np.eye(L)[None]
            rhs = np.concatenate([bc[:, :, None] * Vc,
                                  (bc * np.exp(G))[:, :, None] * Kc], axis=2)
            X = np.linalg.solve(I + A, rhs)
            Ut, W = X[:, :, :Dv], X[:, :, Dv:]
            U = Ut - W @ S
            QK = Qc @ np.transpose(Kc, (0, 2, 1))
            Oc = np.exp(G)[:, :, None] * (Qc @ S) + (dec * QK) @ U
            if keep is None:
                o[c0:c1] = np.transpose(Oc, (1, 0, 2))
            else:
                rows = np.nonzero(keep[c0:c1])[0]
                if rows.size:
                    o[c0 + rows] = np.transpose(Oc[:, rows], (1, 0, 2))
            GL = G[:, -1]
            Kd = np.exp(GL[:, None] - G)[:, :, None] * Kc
            S = np.exp(GL)[:, None, None] * S + np.transpose(Kd, (0, 2, 1)) @ U
        finals[s] = S
    return o, finals


# ---------------------------------------------------------------------------
# a6: gated RMSNorm
# ---------------------------------------------------------------------------

def gated_rmsnorm(x, z, w, eps=1e-6):
    """y = x / sqrt(mean(x^2) + eps) * w * silu(z) over the last axis."""
    x = _f64(x)
    rms = np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return x / rms * _f64(w) * silu(z)


# ---------------------------------------------------------------------------
# a7: one decode step of the whole mixer (one token per sequence)
# ---------------------------------------------------------------------------

def decode_step(mixed_qkv, conv_w, conv_state, a, b, A_log, dt_bias, state, z,
                norm_w, Nk, Nv, Dk, Dv, conv_bias=None, q_scale=None,
                l2_eps=1e-6, norm_eps=1e-6):
    """conv update + SiLU + split/L2/scale + gating + one recurrent step + gated
    RMSNorm, for B sequences with one new token each.

    mixed_qkv [B, C]; conv_state [B, C, K-1]; a, b [B, Nv]; state
    [B, Nv, Dk, Dv]; z [B, Nv, Dv].  Returns dict y [B, Nv, Dv], state,
    conv_state (the updated copies).
    """
    B = mixed_qkv.shape[0]
    cg = conv_gating(mixed_qkv, conv_w, a, b, A_log, dt_bias, Nk, Nv, Dk, Dv,
                     cu_seqlens=None, num_seqs=B, conv_bias=conv_bias,
                     conv_state=conv_state, q_scale=q_scale, l2_eps=l2_eps)
    o, S = recurrent_gated_delta_rule(cg['q'], cg['k'], cg['v'], cg['g'], cg['beta'],
                                      1.0, state, None, B)
    y = gated_rmsnorm(o, z, norm_w, norm_eps)
    return dict(y=y, state=S, conv_state=cg['conv_state'], o=o)


def mixer_prefill(mixed_qkv, conv_w, a, b, A_log, dt_bias, z, norm_w, Nk, Nv, Dk, Dv,
                  cu_seqlens=None, num_seqs=1, conv_bias=None, conv_state=None,
                  initial_state=None, q_scale=None, l2_eps=1e-6, norm_eps=1e-6,
                  use_chunked=False, keep=None):
    """Prefill of the whole mixer: conv_gating -> delta rule -> gated RMSNorm."""
    cg = conv_gating(mixed_qkv, conv_w, a, b, A_log, dt_bias, Nk, Nv, Dk, Dv,
                     cu_seqlens=cu_seqlens, num_seqs=num_seqs, conv_bias=conv_bias,
                     conv_state=conv_state, q_scale=q_scale, l2_eps=l2_eps)
    if use_chunked:
        o, S = chunk_gated_delta_rule(cg['q'], cg['k'], cg['v'], cg['g'], cg['beta'],
                                      1.0, initial_state, cu_seqlens, num_seqs, keep=keep)
    else:
        o, S = recurrent_gated_delta_rule(cg['q'], cg['k'], cg['v'], cg['g'], cg['beta'],
                                          1.0, initial_state, cu_seqlens, num_seqs)
    y = gated_rmsnorm(o, z, norm_w, norm_eps)
    return dict(y=y, o=o, state=S, conv_state=cg['conv_state'], q=cg['q'], k=cg['k'],
                v=cg['v'], g=cg['g'], beta=cg['beta'])
