"""Helpers shared by the GPU parity tests: run the fp64 oracle and the CUDA
path on the same seeded inputs and compare element by element.

Tolerances (stated for the GDN core: bf16 outputs max_abs <= 2e-2 and
mean_abs <= 2e-3; fp32 final states max_abs <= 5e-3; decode state update
within 1e-4 relative).  Readings of those bounds, written out here:
  * outputs are bf16, so each element carries its own rounding of up to half
    a bf16 ulp (<= 2^-8 |x|).  The max bound is applied to the error in excess
    of that representation limit: |gpu - ref| <= 2e-2 + 2^-8 |ref|.  The plain
    max_abs is still reported.  (Only the gated-RMSNorm outputs, which reach
    |y| ~ 10, come near the difference.)
  * "1e-4 relative" for the decode state is max|S_gpu - S_ref| / max|S_ref|
    per step (element-wise relative error is meaningless near zero).
  * the extra weak-decay cases (not among the five workloads) let the state
    grow well above 1; their state bound scales as 5e-3 * max(1, max|S_ref|).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from gated_deltanet_linear_08_gb300.inputs import to_f64

OUT_MAX = 2e-2
OUT_MEAN = 2e-3
STATE_MAX = 5e-3
DECODE_STATE_REL = 1e-4
BF16_HALF_ULP_REL = 2.0 ** -8


def oracle_prefill(x, nthreads: int = 0):
    f = {k: to_f64(x[k]) for k in ("q", "k", "v", "a", "b", "A_log", "dt_bias", "init_state",
                                    "z", "norm_w")}
    return oracle.prefill(x["cu_seqlens"].numpy(), f["q"], f["k"], f["v"], f["a"], f["b"],
                          f["A_log"], f["dt_bias"], f["init_state"], f["z"], f["norm_w"],
                          eps=x["eps"], nthreads=nthreads)


def to_dev(x, dev="cuda"):
    d = {}
    for k in ("q", "k", "v", "a", "b", "A_log", "dt_bias", "init_state", "cu_seqlens", "z",
              "norm_w"):
        d[k] = None if x[k] is None else x[k].to(dev).contiguous()
    return d


def gpu_prefill(x, dev="cuda", in_place=False, stream=None):
    import gated_deltanet_linear_08_gb300 as gdn
    d = to_dev(x, dev)
    fin = d["init_state"] if (in_place and d["init_state"] is not None) else None
    out, fin = gdn.prefill(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                           d["cu_seqlens"], init_state=d["init_state"], z=d["z"],
                           norm_w=d["norm_w"], eps=x["eps"], final_state=fin, stream=stream)
    torch.cuda.synchronize()
    assert gdn.check_device_status() == 0
    return out.double().cpu().numpy(), fin.double().cpu().numpy()


# Every comparison made through assert_out_close / assert_state_close (and
# the decode runs) is recorded here; with GDN_PARITY_REPORT=<path> in the
# environment, tests/conftest.py writes them out as a markdown table at the
# end of the session.
RECORDS = []


def record(what, kind, stats, bound=None):
    RECORDS.append(dict(what=what, kind=kind, bound=bound, **stats))


def out_stats(got, ref):
    err = np.abs(got - ref)
    excess = err - BF16_HALF_ULP_REL * np.abs(ref)
    return dict(max_abs=float(err.max(initial=0.0)), mean_abs=float(err.mean()) if err.size else 0.0,
                p99_abs=float(np.percentile(err, 99)) if err.size else 0.0,
                max_excess=float(excess.max(initial=-1.0)),
                violations=int((excess > OUT_MAX).sum()))


def state_stats(got, ref, bound=STATE_MAX):
    err = np.abs(got - ref)
    return dict(max_abs=float(err.max(initial=0.0)), mean_abs=float(err.mean()) if err.size else 0.0,
                p99_abs=float(np.percentile(err, 99)) if err.size else 0.0,
                violations=int((err > bound).sum()))


def assert_out_close(got, ref, what="out"):
    s = out_stats(got, ref)
    record(what, "out", s, f"excess <= {OUT_MAX:g}, mean <= {OUT_MEAN:g}")
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    assert s["violations"] == 0 and s["mean_abs"] <= OUT_MEAN, f"{what}: {s}"
    return s


def assert_state_close(got, ref, what="state", scale_with_ref=False):
    ref_max = float(np.abs(ref).max(initial=0.0))
    bound = STATE_MAX * (max(1.0, ref_max) if scale_with_ref else 1.0)
    s = state_stats(got, ref, bound)
    s["ref_max_abs"] = ref_max
    record(what, "state", s, f"max <= {bound:.3g}")
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    assert s["violations"] == 0, f"{what}: bound {bound}: {s}"
    return s


# ---------------------------------------------------------------------------
# The causal conv ahead of the core rounds its output to bf16.  The kernels
# evaluate it in fp32 (exact bf16 products, fp32 fma sums, fast exp and
# divide in the SiLU), the oracle in fp64, so where the exact value lies
# within the fp32 evaluation error of a bf16 rounding midpoint the two may
# round apart.  Both are correct roundings: the result of the conv is not
# unique there.  The parity tests therefore (1) check that every conv output
# the GPU produced is a valid rounding of the exact value, and count those
# that differ from the oracle's own rounding, then (2) run the oracle's core
# on the GPU's conv outputs and hold the GPU's core to the usual bounds.
#
# The fp32 evaluation error: the K-1 fmas each add at most 2^-24 of the
# running sum (|partial sums| <= M = sum_j |w_j x_j|), the SiLU (slope <= 1.1)
# carries that through and adds a few fp32 ulps of its own from the fast
# exponential and divide.  2^-20 (|y| + M) bounds the total with margin (it is
# 5x above (K-1) 1.1 2^-24 M + 2^-21 |y| at K = 4).
CONV_ERR_REL = 2.0 ** -20


def conv_exact(x, w, state):
    """The conv's exact (unrounded, fp64) outputs and magnitude sums for one
    sequence: x [T, C] raw inputs, w [C, K], state [K-1, C] or None.  Used
    only to decide which roundings are valid; the reference roundings come
    from oracle.causal_conv_silu."""
    T, C = x.shape
    K = w.shape[1]
    prev = np.zeros((K - 1, C)) if state is None else state
    xe = np.concatenate([prev, x], axis=0)
    terms = np.stack([w[None, :, j] * xe[j:j + T] for j in range(K)], axis=-1)   # [T, C, K]
    return oracle.silu(terms.sum(axis=-1)), np.abs(terms).sum(axis=-1)


def bf16_ulp(y):
    _, e = np.frexp(np.abs(y))
    return np.ldexp(1.0, e - 8)   # bf16 carries 8 significant bits


def conv_check_rounding(got, x, w, state):
    """got: the GPU's conv outputs of one sequence [T, C] (bf16 values as fp64).
    Every element must lie within half a bf16 ulp of the exact value plus the
    fp32 evaluation bound.  Returns the number of elements that differ from
    the oracle's rounding (ties rounded the other way); raises on an invalid
    one."""
    y, mag = conv_exact(x, w, state)
    ref, _ = oracle.causal_conv_silu(x, w, state)
    assert np.all(np.isfinite(got)), "non-finite conv output"
    ulp = bf16_ulp(np.maximum(np.abs(y), np.abs(got)))
    bad = np.abs(got - y) > 0.5 * ulp + CONV_ERR_REL * (np.abs(y) + mag)
    if bad.any():
        t, c = np.argwhere(bad)[0]
        raise AssertionError(f"{int(bad.sum())} invalid conv roundings, first at token {t} channel {c}: "
                             f"got {got[t, c]!r}, exact {y[t, c]!r}, oracle {ref[t, c]!r}")
    return int((got != ref).sum())


def split_qkv(X, hk, hv, d=128):
    T = X.shape[0]
    return (X[:, :hk * d].reshape(T, hk, d).contiguous(), X[:, hk * d:2 * hk * d].reshape(T, hk, d).contiguous(),
            X[:, 2 * hk * d:].reshape(T, hv, d).contiguous())
