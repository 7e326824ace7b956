"""Planted mistakes in the oracle fail its pins (CPU only).

Each mutant is the oracle's C source with one plausible slip: a flipped
sign, a dropped term, a wrong index or operand, a misplaced epsilon, a wrong
head mapping.  It is compiled to a library of its own, the pins of
tests/test_oracle.py run on it, and at least one of them must fail.  A copy
of the source with no change, built the same way, must pass them all, so a
failure means the pins saw the slip and not the harness.

The recurrence the pins fix is the gated delta rule whose ingredients the
JevAny page lists ("Add opt-in fused Qwen3.5 inference kernels", Summary):
gate from A_log and dt_bias, beta sigmoid, q/k L2 norm, grouped value heads,
fused gated RMSNorm.  Every mutant keeps its memory accesses in bounds.
"""
import pytest

import oracle
import test_oracle as pins

# (name, text in gdn_oracle.c, replacement); the first occurrence is replaced
MUTANTS = [
    ("gate_sign",
     "g[t * hv + h] = -exp(A_log[h]) * gdn_oracle_softplus(x);",
     "g[t * hv + h] = exp(A_log[h]) * gdn_oracle_softplus(x);"),
    ("gate_without_dt_bias",
     "double x = a[t * hv + h] + dt_bias[h];",
     "double x = a[t * hv + h];"),
    ("gate_without_exp_A_log",
     "g[t * hv + h] = -exp(A_log[h]) * gdn_oracle_softplus(x);",
     "g[t * hv + h] = -A_log[h] * gdn_oracle_softplus(x);"),
    ("softplus_without_one",
     "    return log1p(exp(x));",
     "    return log(exp(x));"),
    ("sigmoid_sign",
     "return 1.0 / (1.0 + exp(-x));",
     "return 1.0 / (1.0 + exp(x));"),
    ("l2_eps_outside_sqrt",
     "double rq = 1.0 / sqrt(sq + l2_eps), rk = 1.0 / sqrt(sk + l2_eps);",
     "double rq = 1.0 / (sqrt(sq) + l2_eps), rk = 1.0 / (sqrt(sk) + l2_eps);"),
    ("q_scaled_by_k_norm",
     "qn[(t * hk + h) * dk + i] = qs[i] * rq;",
     "qn[(t * hk + h) * dk + i] = qs[i] * rk;"),
    ("no_decay",
     "                S[e] *= eg;",
     "                S[e] *= 1.0;"),
    ("delta_sign",
     "kv[j] = bt * (vt[j] - acc);",
     "kv[j] = bt * (vt[j] + acc);"),
    ("delta_without_beta",
     "kv[j] = bt * (vt[j] - acc);",
     "kv[j] = (vt[j] - acc);"),
    ("output_reads_k",
     "                    acc += S[(size_t)i * dv + j] * qt[i];",
     "                    acc += S[(size_t)i * dv + j] * kt[i];"),
    ("output_without_scale",
     "                ot[j] = acc * scale;",
     "                ot[j] = acc;"),
    ("head_map_modulo",
     "const int n = (int)(u / hv), h = (int)(u % hv), hq = h / group;\n        double *S",
     "const int n = (int)(u / hv), h = (int)(u % hv), hq = h % hk;\n        double *S"),
    ("init_state_by_sequence",
     "memcpy(S, init_state + (size_t)u * ssz, sizeof(double) * ssz);\n        else\n            memset(S, 0, sizeof(double) * ssz);\n        for (int64_t t",
     "memcpy(S, init_state + (size_t)n * ssz, sizeof(double) * ssz);\n        else\n            memset(S, 0, sizeof(double) * ssz);\n        for (int64_t t"),
    ("first_token_skipped",
     "for (int64_t t = cu[n]; t < cu[n + 1]; ++t) {",
     "for (int64_t t = cu[n] + 1; t < cu[n + 1]; ++t) {"),
    ("norm_sum_not_mean",
     "double r = 1.0 / sqrt(ss / dv + eps);",
     "double r = 1.0 / sqrt(ss + eps);"),
    ("norm_gate_sigmoid_only",
     "(z[j] * gdn_oracle_sigmoid(z[j]))",
     "gdn_oracle_sigmoid(z[j])"),
    ("norm_without_weight",
     "o[j] = o[j] * r * w[j] *",
     "o[j] = o[j] * r *"),
]

# pins that run on every mutant (fast cases of the parametrized ones)
PINS = [
    (pins.test_golden_tiny_core_by_hand, {}),
    (pins.test_golden_gated_rmsnorm_by_hand, {}),
    (pins.test_softplus_sigmoid_match_library_on_grid, {}),
    (pins.test_prep_gate_beta_and_l2norm, {}),
    (pins.test_single_token_from_zero_state, {"dk": 4, "dv": 7}),
    (pins.test_beta_zero_is_pure_decay, {}),
    (pins.test_exact_replacement_with_basis_keys, {}),
    (pins.test_dense_brute_force, {"dk": 8, "dv": 3, "T": 7, "unit_keys": False}),
    (pins.test_grouped_heads_use_contiguous_groups, {}),
    (pins.test_chunked_matches_token_form, {"T": 65}),
    (pins.test_split_sequence_with_carried_state_is_bitwise, {}),
    (pins.test_varlen_packing_equals_each_sequence_alone, {}),
    (pins.test_gated_rmsnorm_unit_rms_invariant, {}),
    (pins.test_prefill_is_prep_then_core_then_norm, {}),
    (pins.test_decode_step_equals_one_token_prefill_and_one_pass_identity, {}),
]


def _failing_pins(tmp_path, source):
    src = tmp_path / "gdn_oracle_copy.c"
    src.write_text(source)
    lib = oracle.build(force=True, src=str(src), out=str(tmp_path / "libgdn_oracle_copy.so"))
    failed = []
    with oracle.library(lib):
        for fn, kw in PINS:
            try:
                fn(**kw)
            except AssertionError:
                failed.append(fn.__name__)
    return failed


def _source():
    with open(oracle._SRC) as f:
        return f.read()


def test_unchanged_copy_passes_every_pin(tmp_path):
    assert _failing_pins(tmp_path, _source()) == []


@pytest.mark.parametrize("name,find,repl", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(tmp_path, name, find, repl):
    src = _source()
    assert find in src, f"mutation site of {name} not found"
    failed = _failing_pins(tmp_path, src.replace(find, repl, 1))
    assert failed, f"the oracle with '{name}' planted passes every pin"
    print(name, "caught by", failed)


# ---------------------------------------------------------------------------
# The conv half of the oracle is Python (oracle/__init__.py): a mutated copy
# of the module is executed and its conv functions stand in for the real ones
# while the conv pins run.
# ---------------------------------------------------------------------------
CONV_MUTANTS = [
    ("conv_weights_reversed",
     "acc += w[:, j][None, :] * xe[j:j + T]",
     "acc += w[:, K - 1 - j][None, :] * xe[j:j + T]"),
    ("conv_without_silu",
     "return round_bf16(silu(acc)), xe[T:T + K - 1]",
     "return round_bf16(acc), xe[T:T + K - 1]"),
    ("conv_state_ignored",
     "prev = np.zeros((K - 1, C)) if state is None else np.asarray(state, dtype=np.float64)",
     "prev = np.zeros((K - 1, C))"),
    ("conv_new_state_from_the_front",
     "xe[T:T + K - 1] if K > 1",
     "xe[0:K - 1] if K > 1"),
    ("bf16_rounding_truncates",
     "np.rint(m * 256.0) / 256.0",
     "np.trunc(m * 256.0) / 256.0"),
    ("bf16_rounding_seven_bits",
     "np.rint(m * 256.0) / 256.0",
     "np.rint(m * 128.0) / 128.0"),
    ("silu_sign",
     "return x / (1.0 + np.exp(-x))",
     "return x / (1.0 + np.exp(x))"),
    ("conv_channels_k_before_q",
     "qc = y[:, :hk * d].reshape(T, hk, d)\n    kc = y[:, hk * d:2 * hk * d].reshape(T, hk, d)",
     "kc = y[:, :hk * d].reshape(T, hk, d)\n    qc = y[:, hk * d:2 * hk * d].reshape(T, hk, d)"),
]

CONV_PINS = [
    pins.test_round_bf16_matches_torch_for_fp32_values,
    pins.test_conv_impulse_weights_give_silu_and_shifts,
    pins.test_conv_matches_numpy_convolve_per_channel,
    pins.test_conv_split_sequence_carries_the_state,
    pins.test_conv_inputs_channel_order_is_q_k_v,
]
CONV_FUNCS = ("round_bf16", "silu", "causal_conv_silu", "conv_inputs")


def _failing_conv_pins(monkeypatch, source):
    import types
    mod = types.ModuleType("oracle_copy")
    mod.__file__ = oracle.__file__
    exec(compile(source, "oracle_copy", "exec"), mod.__dict__)
    for f in CONV_FUNCS:
        monkeypatch.setattr(oracle, f, getattr(mod, f))
    failed = []
    for fn in CONV_PINS:
        try:
            fn()
        except Exception:   # an assertion, or a mistake that breaks the shapes
            failed.append(fn.__name__)
    return failed


def _py_source():
    with open(oracle.__file__) as f:
        return f.read()


def test_unchanged_conv_copy_passes_every_conv_pin(monkeypatch):
    assert _failing_conv_pins(monkeypatch, _py_source()) == []


@pytest.mark.parametrize("name,find,repl", CONV_MUTANTS, ids=[m[0] for m in CONV_MUTANTS])
def test_planted_conv_mistake_fails_a_pin(monkeypatch, name, find, repl):
    src = _py_source()
    assert find in src, f"mutation site of {name} not found"
    failed = _failing_conv_pins(monkeypatch, src.replace(find, repl, 1))
    assert failed, f"the conv oracle with '{name}' planted passes every conv pin"
    print(name, "caught by", failed)
