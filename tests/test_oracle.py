"""Pins for the fp64 oracle (CPU only).

Each test checks the oracle against something other than itself: a worked
example done by hand (tests/golden), closed forms of the gated delta rule,
library routines (numpy/scipy) for the scalar prep, a dense transition-matrix
brute force written independently here, and equivalences the recurrence must
satisfy (chunked vs token form, carried state, varlen packing).

The recurrence being pinned is the gated delta rule whose ingredients the
JevAny page lists ("Add opt-in fused Qwen3.5 inference kernels", Summary) and
whose test methodology the pegainfer page gives ("feat(qwen35): add SM120
FlashInfer GDN prefill candidate", Correctness: FP64 oracle, T = 1, 2, 63,
64, 65, 127, 128 boundaries, chunked vs unchunked prefill).
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
RNG = np.random.default_rng(1234)


def _unit_rows(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _random_core_inputs(rng, seqlens, hk, hv, dk, dv, unit_keys=True, init=True,
                        gate_scale=1.0):
    T = sum(seqlens)
    N = len(seqlens)
    cu = np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int32)
    g = -gate_scale * rng.uniform(0.0, 1.0, size=(T, hv))
    beta = rng.uniform(0.0, 1.0, size=(T, hv))
    qn = rng.standard_normal((T, hk, dk))
    kn = rng.standard_normal((T, hk, dk))
    if unit_keys:
        qn, kn = _unit_rows(qn), _unit_rows(kn)
    v = rng.standard_normal((T, hv, dv))
    S0 = 0.3 * rng.standard_normal((N, hv, dk, dv)) if init else None
    return cu, g, beta, qn, kn, v, S0


# --------------------------------------------------------------------------
# Worked example by hand (exact rationals), tests/golden/tiny_core_d2.json
# --------------------------------------------------------------------------
def test_golden_tiny_core_by_hand():
    with open(os.path.join(HERE, "golden", "tiny_core_d2.json")) as f:
        gold = json.load(f)
    inp = gold["inputs"]
    out, fin = oracle.core(np.array(inp["cu_seqlens"]), np.array(inp["g"]),
                           np.array(inp["beta"]), np.array(inp["qn"]), np.array(inp["kn"]),
                           np.array(inp["v"]), np.array(inp["init_state"]))
    np.testing.assert_allclose(out * math.sqrt(2.0), gold["expected"]["out_times_sqrt2"],
                               rtol=0, atol=1e-14)
    np.testing.assert_allclose(fin, gold["expected"]["final_state"], rtol=0, atol=1e-14)
    # the chunked form reaches the same numbers
    out_c, fin_c = oracle.core_chunked(np.array(inp["cu_seqlens"]), np.array(inp["g"]),
                                       np.array(inp["beta"]), np.array(inp["qn"]),
                                       np.array(inp["kn"]), np.array(inp["v"]),
                                       np.array(inp["init_state"]), chunk=64)
    np.testing.assert_allclose(fin_c, gold["expected"]["final_state"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(out_c, out, rtol=0, atol=1e-14)


def test_golden_gated_rmsnorm_by_hand():
    with open(os.path.join(HERE, "golden", "tiny_core_d2.json")) as f:
        gn = json.load(f)["gated_rmsnorm"]
    y = oracle.gated_rmsnorm(np.array([gn["o"]]), np.array([gn["z"]]), np.array(gn["w"]),
                             gn["eps"])
    want = np.array(gn["expected_over_sqrt2_ln3"]) * math.sqrt(2.0) * math.log(3.0)
    np.testing.assert_allclose(y[0], want, rtol=1e-14, atol=0)


# --------------------------------------------------------------------------
# Scalar prep against library routines and invariants
# --------------------------------------------------------------------------
def test_softplus_sigmoid_match_library_on_grid():
    for x in np.linspace(-60.0, 60.0, 2401):
        sp = oracle.softplus(x)
        ref = float(np.logaddexp(0.0, x))
        assert abs(sp - ref) <= 4e-16 * max(1.0, abs(ref)), (x, sp, ref)
        sg = oracle.sigmoid(x)
        assert abs(sg - float(scipy.special.expit(x))) <= 2e-16, x


def test_prep_gate_beta_and_l2norm():
    T, hk, hv, dk = 37, 2, 6, 128
    q = RNG.standard_normal((T, hk, dk))
    k = 3.0 * RNG.standard_normal((T, hk, dk))
    a = RNG.standard_normal((T, hv))
    b = RNG.standard_normal((T, hv))
    A_log = np.log(RNG.uniform(1.0, 16.0, size=hv))
    dt_bias = RNG.standard_normal(hv)
    g, beta, qn, kn = oracle.prep(q, k, a, b, A_log, dt_bias, l2_eps=1e-6)
    # gate: -exp(A_log) * softplus(a + dt_bias), softplus from numpy's logaddexp
    want_g = -np.exp(A_log)[None, :] * np.logaddexp(0.0, a + dt_bias[None, :])
    np.testing.assert_allclose(g, want_g, rtol=1e-14)
    assert np.all(g < 0)
    np.testing.assert_allclose(beta, scipy.special.expit(b), rtol=1e-15)
    # L2 norm: unit length up to the epsilon inside the root, same direction
    for x, xn in ((q, qn), (k, kn)):
        nrm = np.linalg.norm(x, axis=-1)
        np.testing.assert_allclose(np.linalg.norm(xn, axis=-1),
                                   nrm / np.sqrt(nrm ** 2 + 1e-6), rtol=1e-14)
        cos = np.sum(x * xn, axis=-1) / (nrm * np.linalg.norm(xn, axis=-1))
        np.testing.assert_allclose(cos, 1.0, rtol=1e-14)
    # the special point a + dt_bias = 0, A_log = 0 gives g = -ln 2 and b = 0 gives 1/2
    g0, b0, _, _ = oracle.prep(q[:1], k[:1], np.zeros((1, 1)), np.zeros((1, 1)),
                               np.zeros(1), np.zeros(1))
    assert abs(g0[0, 0] + math.log(2.0)) < 1e-15 and b0[0, 0] == 0.5


def test_prep_zero_vector_stays_finite():
    z = np.zeros((1, 1, 128))
    _, _, qn, kn = oracle.prep(z, z, np.zeros((1, 1)), np.zeros((1, 1)), np.zeros(1),
                               np.zeros(1))
    assert np.all(qn == 0) and np.all(kn == 0)


# --------------------------------------------------------------------------
# Closed forms of the recurrence
# --------------------------------------------------------------------------
@pytest.mark.parametrize("dk,dv", [(128, 128), (4, 7)])
def test_single_token_from_zero_state(dk, dv):
    cu, g, beta, qn, kn, v, _ = _random_core_inputs(RNG, [1], 1, 1, dk, dv, init=False)
    out, fin = oracle.core(cu, g, beta, qn, kn, v, None)
    b0 = beta[0, 0]
    np.testing.assert_allclose(fin[0, 0], b0 * np.outer(kn[0, 0], v[0, 0]), atol=1e-15)
    want_o = b0 * float(kn[0, 0] @ qn[0, 0]) * v[0, 0] / math.sqrt(dk)
    np.testing.assert_allclose(out[0, 0], want_o, atol=1e-15)


def test_beta_zero_is_pure_decay():
    dk, dv, T = 16, 8, 9
    cu, g, beta, qn, kn, v, S0 = _random_core_inputs(RNG, [T], 1, 1, dk, dv)
    beta[:] = 0.0
    out, fin = oracle.core(cu, g, beta, qn, kn, v, S0)
    G = np.cumsum(g[:, 0])
    np.testing.assert_allclose(fin[0, 0], math.exp(G[-1]) * S0[0, 0], rtol=1e-13)
    for t in range(T):
        want = math.exp(G[t]) * (S0[0, 0].T @ qn[t, 0]) / math.sqrt(dk)
        np.testing.assert_allclose(out[t, 0], want, rtol=1e-12, atol=1e-15)


def test_exact_replacement_with_basis_keys():
    """g = 0, beta = 1, keys = distinct basis vectors: each written row is
    replaced exactly and the rest of the state is untouched."""
    dk, dv = 8, 5
    idx = [3, 0, 6, 1]
    T = len(idx)
    cu = np.array([0, T], dtype=np.int32)
    g = np.zeros((T, 1))
    beta = np.ones((T, 1))
    kn = np.zeros((T, 1, dk))
    for t, i in enumerate(idx):
        kn[t, 0, i] = 1.0
    qn = _unit_rows(RNG.standard_normal((T, 1, dk)))
    v = RNG.standard_normal((T, 1, dv))
    S0 = RNG.standard_normal((1, 1, dk, dv))
    out, fin = oracle.core(cu, g, beta, qn, kn, v, S0)
    want = S0[0, 0].copy()
    for t, i in enumerate(idx):
        want[i, :] = v[t, 0]
    np.testing.assert_allclose(fin[0, 0], want, rtol=0, atol=1e-15)
    for t, i in enumerate(idx):
        np.testing.assert_allclose(fin[0, 0].T @ kn[t, 0], v[t, 0], atol=1e-15)


# --------------------------------------------------------------------------
# Dense brute force on tiny T: S_T = (prod A_t) S0 + sum_s (prod_{r>s} A_r) beta_s k_s v_s^T
# with A_t = e^{g_t} (I - beta_t k_t k_t^T), built as explicit Dk x Dk matrices.
# --------------------------------------------------------------------------
def _brute_force(g, beta, qn, kn, v, S0, dk):
    T = g.shape[0]
    trans = [math.exp(g[t]) * (np.eye(dk) - beta[t] * np.outer(kn[t], kn[t]))
             for t in range(T)]
    states = []
    for t in range(T):
        # prod_{r<=t} A_r applied in time order: A_t ... A_0
        M = np.eye(dk)
        for r in range(t + 1):
            M = trans[r] @ M
        St = M @ S0
        for s in range(t + 1):
            Ms = np.eye(dk)
            for r in range(s + 1, t + 1):
                Ms = trans[r] @ Ms
            St = St + Ms @ (beta[s] * np.outer(kn[s], v[s]))
        states.append(St)
    outs = np.stack([states[t].T @ qn[t] / math.sqrt(dk) for t in range(T)])
    return outs, states[-1]


@pytest.mark.parametrize("dk,dv,T", [(4, 4, 8), (8, 3, 7), (128, 128, 5), (5, 9, 1)])
@pytest.mark.parametrize("unit_keys", [True, False])
def test_dense_brute_force(dk, dv, T, unit_keys):
    cu, g, beta, qn, kn, v, S0 = _random_core_inputs(RNG, [T], 1, 1, dk, dv,
                                                     unit_keys=unit_keys)
    out, fin = oracle.core(cu, g, beta, qn, kn, v, S0)
    bo, bs = _brute_force(g[:, 0], beta[:, 0], qn[:, 0], kn[:, 0], v[:, 0], S0[0, 0], dk)
    np.testing.assert_allclose(fin[0, 0], bs, rtol=0, atol=1e-12 * max(1, np.abs(bs).max()))
    np.testing.assert_allclose(out[:, 0], bo, rtol=0, atol=1e-12 * max(1, np.abs(bo).max()))


def test_grouped_heads_use_contiguous_groups():
    """Hv/Hk = 3: value head h reads key/query head h // 3 (reading of 'grouped
    value heads'); checked per head against the brute force."""
    hk, hv, dk, dv, T = 2, 6, 6, 4, 5
    cu, g, beta, qn, kn, v, S0 = _random_core_inputs(RNG, [T], hk, hv, dk, dv)
    out, fin = oracle.core(cu, g, beta, qn, kn, v, S0)
    for h in range(hv):
        hq = h // 3
        bo, bs = _brute_force(g[:, h], beta[:, h], qn[:, hq], kn[:, hq], v[:, h],
                              S0[0, h], dk)
        np.testing.assert_allclose(fin[0, h], bs, atol=1e-12)
        np.testing.assert_allclose(out[:, h], bo, atol=1e-12)


# --------------------------------------------------------------------------
# Equivalences
# --------------------------------------------------------------------------
@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 127, 128, 200])
def test_chunked_matches_token_form(T):
    cu, g, beta, qn, kn, v, S0 = _random_core_inputs(RNG, [T], 1, 2, 16, 8)
    out, fin = oracle.core(cu, g, beta, qn, kn, v, S0)
    out_c, fin_c = oracle.core_chunked(cu, g, beta, qn, kn, v, S0, chunk=64)
    np.testing.assert_allclose(out_c, out, rtol=0, atol=1e-10)
    np.testing.assert_allclose(fin_c, fin, rtol=0, atol=1e-10)


def test_chunked_matches_token_form_weak_decay_full_width():
    cu, g, beta, qn, kn, v, S0 = _random_core_inputs(RNG, [150], 1, 1, 128, 128,
                                                     gate_scale=0.01)
    out, fin = oracle.core(cu, g, beta, qn, kn, v, S0)
    for C in (16, 64):
        out_c, fin_c = oracle.core_chunked(cu, g, beta, qn, kn, v, S0, chunk=C)
        np.testing.assert_allclose(out_c, out, rtol=0, atol=1e-10)
        np.testing.assert_allclose(fin_c, fin, rtol=0, atol=1e-10)


def test_split_sequence_with_carried_state_is_bitwise():
    T = 23
    cu, g, beta, qn, kn, v, S0 = _random_core_inputs(RNG, [T], 1, 2, 8, 6)
    out, fin = oracle.core(cu, g, beta, qn, kn, v, S0)
    for m in range(0, T + 1):
        c1 = np.array([0, m], dtype=np.int32)
        c2 = np.array([0, T - m], dtype=np.int32)
        o1, f1 = oracle.core(c1, g[:m], beta[:m], qn[:m], kn[:m], v[:m], S0)
        o2, f2 = oracle.core(c2, g[m:], beta[m:], qn[m:], kn[m:], v[m:], f1)
        assert np.array_equal(np.concatenate([o1, o2]), out)
        assert np.array_equal(f2, fin)


def test_varlen_packing_equals_each_sequence_alone():
    seqlens = [5, 1, 0, 17, 64, 3]
    cu, g, beta, qn, kn, v, S0 = _random_core_inputs(RNG, seqlens, 2, 4, 8, 8)
    out, fin = oracle.core(cu, g, beta, qn, kn, v, S0)
    for n in range(len(seqlens)):
        s, e = cu[n], cu[n + 1]
        o1, f1 = oracle.core(np.array([0, e - s], dtype=np.int32), g[s:e], beta[s:e],
                             qn[s:e], kn[s:e], v[s:e], S0[n:n + 1])
        assert np.array_equal(o1, out[s:e])
        assert np.array_equal(f1[0], fin[n])
    # an empty sequence hands its initial state through unchanged
    assert np.array_equal(fin[2], S0[2])


def test_gated_rmsnorm_unit_rms_invariant():
    o = RNG.standard_normal((50, 128))
    z = RNG.standard_normal((50, 128))
    w = 1.0 + 0.1 * RNG.standard_normal(128)
    eps = 1e-6
    y = oracle.gated_rmsnorm(o, z, w, eps)
    gate = w[None, :] * z * scipy.special.expit(z)
    r = y / gate
    ms = np.mean(r ** 2, axis=-1)
    want = np.mean(o ** 2, axis=-1) / (np.mean(o ** 2, axis=-1) + eps)
    np.testing.assert_allclose(ms, want, rtol=1e-12)


def test_prefill_is_prep_then_core_then_norm():
    from gated_deltanet_linear_08_gb300.inputs import PrefillCase, make_prefill_inputs, to_f64
    case = PrefillCase("t", seqlens=[7, 70], hk=2, hv=4, init_state=True, gated_norm=True)
    x = make_prefill_inputs(case)
    f = {k: to_f64(x[k]) for k in ("q", "k", "v", "a", "b", "A_log", "dt_bias",
                                    "init_state", "z", "norm_w")}
    out, fin = oracle.prefill(x["cu_seqlens"].numpy(), f["q"], f["k"], f["v"], f["a"],
                              f["b"], f["A_log"], f["dt_bias"], f["init_state"], f["z"],
                              f["norm_w"], eps=x["eps"])
    g, beta, qn, kn = oracle.prep(f["q"], f["k"], f["a"], f["b"], f["A_log"], f["dt_bias"])
    o2, f2 = oracle.core(x["cu_seqlens"].numpy(), g, beta, qn, kn, f["v"], f["init_state"])
    y2 = oracle.gated_rmsnorm(o2, f["z"], f["norm_w"], x["eps"])
    assert np.array_equal(out, y2) and np.array_equal(fin, f2)


def test_decode_step_equals_one_token_prefill_and_one_pass_identity():
    """Decode = the same body with T = 1.  Also pins the single-read identity a
    streaming decode kernel uses: with r_k, r_q read from the OLD state,
    delta = beta (v - e^g r_k) and o = scale (e^g r_q + (k.q) delta) equal
    scale * S_new^T q exactly (up to rounding)."""
    B, hk, hv, dk = 3, 2, 4, 128
    q = RNG.standard_normal((B, hk, dk)); k = RNG.standard_normal((B, hk, dk))
    v = RNG.standard_normal((B, hv, dk))
    a = RNG.standard_normal((B, hv)); b = RNG.standard_normal((B, hv))
    A_log = np.log(RNG.uniform(1, 16, hv)); dt_bias = RNG.standard_normal(hv)
    S = 0.1 * RNG.standard_normal((B, hv, dk, dk))
    S_old = S.copy()
    out = oracle.decode_step(q, k, v, a, b, A_log, dt_bias, S)
    g, beta, qn, kn = oracle.prep(q, k, a, b, A_log, dt_bias)
    scale = 1.0 / math.sqrt(dk)
    for n in range(B):
        for h in range(hv):
            hq = h // (hv // hk)
            eg = math.exp(g[n, h])
            rk = S_old[n, h].T @ kn[n, hq]
            rq = S_old[n, h].T @ qn[n, hq]
            delta = beta[n, h] * (v[n, h] - eg * rk)
            o1 = scale * (eg * rq + float(kn[n, hq] @ qn[n, hq]) * delta)
            np.testing.assert_allclose(out[n, h], o1, rtol=0, atol=1e-14)
            np.testing.assert_allclose(S[n, h], eg * S_old[n, h] + np.outer(kn[n, hq], delta),
                                       rtol=0, atol=1e-15)


def test_multi_token_decode_equals_recurrence_over_the_draft():
    """Decoding T tokens of one sequence in a row (a speculative draft) is the
    recurrence over those T tokens from the sequence's state: T successive
    oracle decode steps equal the token-by-token core over a T-token sequence
    with that initial state, outputs and final state."""
    T, hk, hv, dk = 5, 2, 4, 128
    q = RNG.standard_normal((T, hk, dk)); k = RNG.standard_normal((T, hk, dk))
    v = RNG.standard_normal((T, hv, dk))
    a = RNG.standard_normal((T, hv)); b = RNG.standard_normal((T, hv))
    A_log = np.log(RNG.uniform(1, 16, hv)); dt_bias = RNG.standard_normal(hv)
    S0 = 0.1 * RNG.standard_normal((1, hv, dk, dk))
    S = S0.copy()
    outs = [oracle.decode_step(q[t:t + 1], k[t:t + 1], v[t:t + 1], a[t:t + 1], b[t:t + 1],
                               A_log, dt_bias, S)[0] for t in range(T)]
    g, beta, qn, kn = oracle.prep(q, k, a, b, A_log, dt_bias)
    o2, f2 = oracle.core(np.array([0, T], np.int32), g, beta, qn, kn, v, S0)
    np.testing.assert_allclose(np.stack(outs), o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(S, f2, rtol=0, atol=1e-13)


# --------------------------------------------------------------------------
# causal conv1d + SiLU ahead of the core (a reading: the pages list the
# dependency without defining it)
# --------------------------------------------------------------------------
def test_round_bf16_matches_torch_for_fp32_values():
    import torch
    x = (RNG.standard_normal(4000) * np.exp(RNG.uniform(-8, 8, 4000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.round_bf16(x.astype(np.float64)), ref)


def test_conv_impulse_weights_give_silu_and_shifts():
    T, C, K = 9, 6, 4
    x = oracle.round_bf16(RNG.standard_normal((T, C)))
    st = oracle.round_bf16(RNG.standard_normal((K - 1, C)))
    w = np.zeros((C, K)); w[:, K - 1] = 1.0          # current token only
    y, new = oracle.causal_conv_silu(x, w, st)
    assert np.array_equal(y, oracle.round_bf16(x / (1 + np.exp(-x))))
    assert np.array_equal(new, x[T - (K - 1):])
    w = np.zeros((C, K)); w[:, 0] = 1.0              # the token K-1 steps back
    y, _ = oracle.causal_conv_silu(x, w, st)
    xe = np.concatenate([st, x])
    assert np.array_equal(y, oracle.round_bf16(xe[:T] / (1 + np.exp(-xe[:T]))))
    y0, _ = oracle.causal_conv_silu(x, w, None)      # no state: zeros before the start
    assert np.array_equal(y0[:K - 1], np.zeros((K - 1, C)))


def test_conv_matches_numpy_convolve_per_channel():
    T, C, K = 37, 5, 4
    x = RNG.standard_normal((T, C)); w = RNG.standard_normal((C, K)); st = RNG.standard_normal((K - 1, C))
    y, _ = oracle.causal_conv_silu(x, w, st)
    xe = np.concatenate([st, x])
    for c in range(C):
        acc = np.convolve(xe[:, c], w[c, ::-1], mode="valid")   # a correlation with w
        np.testing.assert_allclose(y[:, c], oracle.round_bf16(acc / (1 + np.exp(-acc))), rtol=0, atol=0)


def test_conv_split_sequence_carries_the_state():
    T, C = 23, 7
    for K in (2, 3, 4):
        x = RNG.standard_normal((T, C)); w = RNG.standard_normal((C, K)); st = RNG.standard_normal((K - 1, C))
        y, new = oracle.causal_conv_silu(x, w, st)
        for cut in (1, 2, 5, 22):
            y1, s1 = oracle.causal_conv_silu(x[:cut], w, st)
            y2, s2 = oracle.causal_conv_silu(x[cut:], w, s1)
            assert np.array_equal(np.concatenate([y1, y2]), y) and np.array_equal(s2, new)


def test_conv_inputs_channel_order_is_q_k_v():
    """The channels are q heads, then k heads, then v heads: weights that pass
    the current token on one block of channels only reproduce exactly that
    input (through SiLU) and leave the other two zero."""
    T, hk, hv, d = 5, 2, 4, 128
    q = RNG.standard_normal((T, hk, d)); k = RNG.standard_normal((T, hk, d)); v = RNG.standard_normal((T, hv, d))
    C = 2 * hk * d + hv * d
    blocks = {"q": (0, hk * d), "k": (hk * d, 2 * hk * d), "v": (2 * hk * d, C)}
    for name, (lo, hi) in blocks.items():
        w = np.zeros((C, 4)); w[lo:hi, 3] = 1.0        # only this block passes the current token
        got = dict(zip("qkv", oracle.conv_inputs(np.array([0, T]), q, k, v, w)[:3]))
        for other, x in (("q", q), ("k", k), ("v", v)):
            want = oracle.round_bf16(x / (1 + np.exp(-x))) if other == name else np.zeros_like(x)
            assert np.array_equal(got[other], want), (name, other)


def test_conv_rounding_check_accepts_an_fp32_evaluation_and_rejects_a_slip():
    """The GPU conv parity accepts, element by element, any valid bf16
    rounding of the exact conv value (parity_util.conv_check_rounding).  An
    independent fp32 evaluation -- torch on the CPU: fp32 sums of the exact
    bf16 products, fp32 SiLU -- on a raw draw passes it, with a few ties
    rounded the other way; the oracle's own rounding passes with none; and a
    copy with one element moved by one bf16 ulp away from any tie fails."""
    import torch
    from parity_util import bf16_ulp, conv_check_rounding, conv_exact
    from gated_deltanet_linear_08_gb300.inputs import make_conv_inputs
    g = torch.Generator().manual_seed(3)
    T, C, K = 96, 512, 4
    X = torch.randn(T, C, generator=g).to(torch.bfloat16)
    cv = make_conv_inputs(C, K, 1, seed=3)
    st = cv["state"][0]
    x64, w64, st64 = X.double().numpy(), cv["weight"].double().numpy(), st.double().numpy()
    y64, _ = oracle.causal_conv_silu(x64, w64, st64)
    xe = torch.cat([st, X]).float()
    w = cv["weight"].float()
    acc = w[:, K - 1] * xe[K - 1:K - 1 + T]
    for j in range(K - 1):
        acc = acc + w[:, j] * xe[j:j + T]
    y32 = (acc * torch.sigmoid(acc)).to(torch.bfloat16).double().numpy()
    flips = conv_check_rounding(y32, x64, w64, st64)
    assert 0 <= flips < 20
    assert conv_check_rounding(y64, x64, w64, st64) == 0
    exact, _ = conv_exact(x64, w64, st64)
    ulp = bf16_ulp(exact)
    far = np.abs(exact - y64) < 0.25 * ulp          # well away from a rounding midpoint
    t, c = np.argwhere(far & (np.abs(exact) > 0.1))[0]
    slip = y64.copy()
    slip[t, c] += ulp[t, c]
    with pytest.raises(AssertionError):
        conv_check_rounding(slip, x64, w64, st64)
