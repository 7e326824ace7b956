"""GPU parity of gdn_decode against the fp64 oracle (one token per sequence,
state updated in place; the recurrent-state slots of the SGLang page "[Perf]
Pack the Qwen3.5 GDN input projection on CUDA", Accuracy Tests).

Every sequence and every step is compared: the outputs element by element
against the bf16 bounds, and the whole state after each step against the
"1e-4 relative" bound (max |S_gpu - S_ref| / max |S_ref|).
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_08_gb300.inputs import CASE_DECODE, DecodeCase, make_decode_inputs, to_f64
from parity_util import DECODE_STATE_REL, OUT_MAX, OUT_MEAN, out_stats, record

pytestmark = pytest.mark.gpu


def _run(case):
    import gated_deltanet_linear_08_gb300 as gdn
    x = make_decode_inputs(case)
    dev = "cuda"
    S_ref = np.ascontiguousarray(to_f64(x["state"]))
    S_dev = x["state"].to(dev)
    A_log, dt = x["A_log"].to(dev), x["dt_bias"].to(dev)
    w = x["norm_w"].to(dev) if x["norm_w"] is not None else None
    worst = dict(max_abs=0.0, mean_abs=0.0, p99_abs=0.0, max_excess=-1.0, violations=0, state_rel=0.0)
    for t, stp in enumerate(x["steps"]):
        z = x["z"][t] if x["z"] is not None else None
        d = {k: v.to(dev) for k, v in stp.items()}
        out = gdn.decode(d["q"], d["k"], d["v"], d["a"], d["b"], A_log, dt, S_dev,
                         z=None if z is None else z.to(dev), norm_w=w, eps=x["eps"])
        ref = oracle.decode_step(*(to_f64(stp[k]) for k in ("q", "k", "v", "a", "b")),
                                 to_f64(x["A_log"]), to_f64(x["dt_bias"]), S_ref,
                                 z=None if z is None else to_f64(z),
                                 norm_w=to_f64(x["norm_w"]), eps=x["eps"])
        got = out.double().cpu().numpy()
        s = out_stats(got, ref)
        assert np.all(np.isfinite(got)) and s["violations"] == 0 and s["mean_abs"] <= OUT_MEAN, (t, s)
        for key in ("max_abs", "p99_abs", "max_excess"):
            worst[key] = max(worst[key], s[key])
        worst["mean_abs"] = max(worst["mean_abs"], s["mean_abs"])
        # the whole state after this step (fp64 difference, on the host cores)
        Sg = S_dev.cpu()
        Sr = torch.from_numpy(S_ref)
        rel = float((Sr - Sg.double()).abs().max() / Sr.abs().max())
        assert rel <= DECODE_STATE_REL, (t, rel)
        worst["state_rel"] = max(worst["state_rel"], rel)
    assert gdn.check_device_status() == 0
    record(f"{case.name}: outputs, worst of {case.steps} steps", "out", {k: worst[k] for k in
           ("max_abs", "mean_abs", "p99_abs", "max_excess", "violations")},
           f"excess <= {OUT_MAX:g}, mean <= {OUT_MEAN:g}")
    record(f"{case.name}: state, worst of {case.steps} steps", "state",
           dict(max_abs=worst["state_rel"], violations=0), f"max|dS|/max|S| <= {DECODE_STATE_REL:g}")
    return worst


def test_decode_small_grouped_heads():
    _run(DecodeCase("decode_small_g3", batch=5, hk=2, hv=6, steps=8))


def test_decode_small_gated_norm():
    _run(DecodeCase("decode_small_gn", batch=3, hk=2, hv=4, steps=6, gated_norm=True))


def test_decode_batch256_64_steps():
    """The full decode workload (B=256, Hk=16, Hv=32, 64 consecutive steps):
    all 256 sequences' outputs and states follow the oracle at every step."""
    w = _run(CASE_DECODE)
    print("decode worst:", w)
