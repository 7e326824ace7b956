"""GPU parity of gdn_decode against the fp64 oracle (one token per sequence,
state updated in place; the recurrent-state slots of the SGLang page "[Perf]
Pack the Qwen3.5 GDN input projection on CUDA", Accuracy Tests).
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_08_gb300.inputs import CASE_DECODE, DecodeCase, make_decode_inputs, to_f64
from parity_util import DECODE_STATE_REL, assert_out_close

pytestmark = pytest.mark.gpu


def _run(case, sample=None, check_every=1):
    import gated_deltanet_linear_08_gb300 as gdn
    x = make_decode_inputs(case)
    dev = "cuda"
    sel = np.arange(case.batch) if sample is None else np.asarray(sample)
    S_ref = np.ascontiguousarray(to_f64(x["state"])[sel])
    S_dev = x["state"].to(dev)
    A_log, dt = x["A_log"].to(dev), x["dt_bias"].to(dev)
    w = x["norm_w"].to(dev) if x["norm_w"] is not None else None
    worst = dict(state_rel=0.0, out_max=0.0)
    for t, stp in enumerate(x["steps"]):
        z = x["z"][t] if x["z"] is not None else None
        d = {k: v.to(dev) for k, v in stp.items()}
        out = gdn.decode(d["q"], d["k"], d["v"], d["a"], d["b"], A_log, dt, S_dev,
                         z=None if z is None else z.to(dev), norm_w=w, eps=x["eps"])
        ref = oracle.decode_step(*(to_f64(stp[k])[sel] for k in ("q", "k", "v", "a", "b")),
                                 to_f64(x["A_log"]), to_f64(x["dt_bias"]), S_ref,
                                 z=None if z is None else to_f64(z)[sel],
                                 norm_w=to_f64(x["norm_w"]), eps=x["eps"])
        got = out.double().cpu().numpy()[sel]
        s = assert_out_close(got, ref, f"decode out step {t}")
        worst["out_max"] = max(worst["out_max"], s["max_abs"])
        if t % check_every == 0 or t == case.steps - 1:
            Sg = S_dev[torch.as_tensor(sel, device=dev)].double().cpu().numpy()
            rel = np.abs(Sg - S_ref).max() / np.abs(S_ref).max()
            assert rel <= DECODE_STATE_REL, (t, rel)
            worst["state_rel"] = max(worst["state_rel"], float(rel))
    assert gdn.check_device_status() == 0
    return worst


def test_decode_small_grouped_heads():
    _run(DecodeCase("small", batch=5, hk=2, hv=6, steps=8))


def test_decode_small_gated_norm():
    _run(DecodeCase("small_gn", batch=3, hk=2, hv=4, steps=6, gated_norm=True))


def test_decode_batch256_64_steps_sampled():
    """The full decode workload (B=256, Hk=16, Hv=32, 64 steps) on the GPU;
    the oracle follows 8 of the 256 sequences (all heads) step by step."""
    w = _run(CASE_DECODE, sample=list(range(0, 256, 32)), check_every=8)
    print("decode worst:", w)
