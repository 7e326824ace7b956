"""The algebra of the multi-token decode kernel, pinned on the CPU in fp64.

A draft of T tokens (T = 2..8) is decoded in one pass over the state: with
G_t the gate summed over the draft's tokens 0..t, Gam_t = e^{G_t},
r_ts = e^{G_t - G_s} and S0 the state before the draft,
    delta_t = beta_t (v_t - Gam_t S0^T k_t) - sum_{s<t} beta_t r_ts (k_s.k_t) delta_s
    o_t     = scale (Gam_t S0^T q_t + sum_{s<=t} r_ts (k_s.q_t) delta_s)
    S_T     = Gam_{T-1} S0 + sum_s (r_{T-1,s} k_s) delta_s^T
This file states that unrolled form in numpy and checks it against the
oracle's one decode step per token (the recurrence itself) to fp64 rounding,
for every draft length the kernel takes, including gates strong enough for
Gam_t to underflow.  The GPU parity tests check the kernel against the same
oracle; this test checks the identity the kernel is built on.
"""
import numpy as np
import pytest

import oracle

D = 16          # head size of these cases (the identity does not depend on it)


def _inputs(rng, T, hk, hv, strong):
    q = rng.standard_normal((T, hk, D))
    k = rng.standard_normal((T, hk, D))
    v = rng.standard_normal((T, hv, D))
    a = rng.standard_normal((T, hv)) * (4.0 if strong else 1.0)
    b = rng.standard_normal((T, hv))
    A_log = np.log(rng.uniform(1.0, 16.0, hv)) + (3.0 if strong else 0.0)
    dt_bias = rng.standard_normal(hv) + (4.0 if strong else 0.0)
    S0 = rng.standard_normal((1, hv, D, D)) * 0.3
    return q, k, v, a, b, A_log, dt_bias, S0


def _unrolled(q, k, v, a, b, A_log, dt_bias, S0):
    """The draft as the kernel solves it (fp64)."""
    T, hk, _ = q.shape
    hv = v.shape[1]
    g, beta, qn, kn = oracle.prep(q, k, a, b, A_log, dt_bias)
    scale = 1.0 / np.sqrt(D)
    out = np.zeros((T, hv, D))
    S_T = np.zeros((hv, D, D))
    for h in range(hv):
        hq = h // (hv // hk)
        K, Q, V, S = kn[:, hq], qn[:, hq], v[:, h], S0[0, h]
        G = np.cumsum(g[:, h])
        r = lambda t, s: np.exp(G[t] - G[s])
        sk, sq = K @ S, Q @ S                     # rows t: S0^T k_t, S0^T q_t
        dl = np.zeros((T, D))
        for t in range(T):
            x = beta[t, h] * (V[t] - np.exp(G[t]) * sk[t])
            for s in range(t):
                x = x - beta[t, h] * r(t, s) * (K[s] @ K[t]) * dl[s]
            dl[t] = x
            o = np.exp(G[t]) * sq[t] + sum(r(t, s) * (K[s] @ Q[t]) * dl[s] for s in range(t + 1))
            out[t, h] = scale * o
        S_T[h] = np.exp(G[-1]) * S + sum(np.outer(r(T - 1, s) * K[s], dl[s]) for s in range(T))
    return out, S_T


def _sequential(q, k, v, a, b, A_log, dt_bias, S0):
    """The oracle's recurrence, one decode step per token."""
    T = q.shape[0]
    S = np.ascontiguousarray(S0.copy())
    out = np.stack([oracle.decode_step(q[t:t + 1], k[t:t + 1], v[t:t + 1], a[t:t + 1], b[t:t + 1],
                                       A_log, dt_bias, S)[0] for t in range(T)])
    return out, S[0]


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("strong", [False, True])
def test_draft_unrolled_form_equals_the_recurrence(T, strong):
    rng = np.random.default_rng(100 * T + strong)
    x = _inputs(rng, T, hk=2, hv=4, strong=strong)
    o1, s1 = _unrolled(*x)
    o2, s2 = _sequential(*x)
    assert np.abs(o1 - o2).max() <= 1e-12 * max(1.0, np.abs(o2).max())
    assert np.abs(s1 - s2).max() <= 1e-12 * max(1.0, np.abs(s2).max())


def test_strong_gates_underflow_and_still_agree():
    """With strong gates the cumulative decay e^{G} of the later tokens
    underflows to zero; the ratios r_ts stay in [0, 1] and the two forms agree."""
    rng = np.random.default_rng(7)
    x = _inputs(rng, 8, hk=2, hv=4, strong=True)
    g, _, _, _ = oracle.prep(x[0], x[1], x[3], x[4], x[5], x[6])
    assert np.exp(np.cumsum(g, axis=0)).min() == 0.0   # some Gam_t underflows
    o1, s1 = _unrolled(*x)
    o2, s2 = _sequential(*x)
    assert np.isfinite(o1).all() and np.isfinite(s1).all()
    assert np.abs(o1 - o2).max() <= 1e-12 * max(1.0, np.abs(o2).max())
    assert np.abs(s1 - s2).max() <= 1e-12 * max(1.0, np.abs(s2).max())
