"""GPU parity of gdn_decode_slots against the fp64 oracle: several consecutive
tokens per sequence (a speculative draft) against a pool of recurrent-state
slots (SGLang page "[Perf] Pack the Qwen3.5 GDN input projection on CUDA",
Accuracy Tests: mamba slots).  The oracle advances each sequence's slot state
through its tokens with one decode step per token.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_08_gb300.inputs import (DecodeCase, DecodeSlotsCase, make_decode_inputs,
                                                   make_decode_slots_inputs, to_f64)
from parity_util import DECODE_STATE_REL, assert_out_close, record

pytestmark = pytest.mark.gpu


def _run(case):
    import gated_deltanet_linear_08_gb300 as gdn
    x = make_decode_slots_inputs(case)
    dev = "cuda"
    B, T, P = case.batch, case.tokens, case.slots
    idx = x["state_idx"].numpy()
    pool_dev = x["pool"].to(dev)
    out = gdn.decode_slots(x["q"].to(dev), x["k"].to(dev), x["v"].to(dev), x["a"].to(dev), x["b"].to(dev),
                           x["A_log"].to(dev), x["dt_bias"].to(dev), pool_dev,
                           state_idx=x["state_idx"].to(dev),
                           z=None if x["z"] is None else x["z"].to(dev),
                           norm_w=None if x["norm_w"] is None else x["norm_w"].to(dev), eps=x["eps"])
    bits = gdn.check_device_status()
    got_out = out.double().cpu().numpy()
    got_pool = pool_dev.cpu()

    live = np.nonzero((idx >= 0) & (idx < P))[0]
    dead = np.nonzero((idx < 0) | (idx >= P))[0]
    # the oracle: the live sequences' slot states, one decode step per token
    S = np.ascontiguousarray(to_f64(x["pool"])[idx[live]])
    ref = np.zeros((len(live), T, case.hv, case.d))
    for t in range(T):
        ref[:, t] = oracle.decode_step(*(to_f64(x[n])[live, t] for n in ("q", "k", "v", "a", "b")),
                                       to_f64(x["A_log"]), to_f64(x["dt_bias"]), S,
                                       z=None if x["z"] is None else to_f64(x["z"])[live, t],
                                       norm_w=to_f64(x["norm_w"]), eps=x["eps"])
    assert_out_close(got_out[live], ref, f"{case.name} out")
    Sg = got_pool[torch.as_tensor(idx[live].astype(np.int64))].double().numpy()
    rel = np.abs(Sg - S).max() / np.abs(S).max()
    record(f"{case.name} state", "state", dict(max_abs=float(rel), violations=int(rel > DECODE_STATE_REL)),
           f"max|dS|/max|S| <= {DECODE_STATE_REL:g}")
    assert rel <= DECODE_STATE_REL, rel
    # skipped sequences: zero outputs; slots nobody named: bitwise untouched
    assert np.all(got_out[dead] == 0)
    untouched = np.setdiff1d(np.arange(P), idx[live])
    assert torch.equal(got_pool[torch.as_tensor(untouched)], x["pool"][torch.as_tensor(untouched)])
    expect_bits = 4 if case.out_of_pool else 0   # the range bit flags indices past the pool
    assert bits == expect_bits, bits
    return rel


@pytest.mark.parametrize("tokens", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("gated", [False, True])
def test_decode_slots_multi_token(tokens, gated):
    _run(DecodeSlotsCase(f"slots_T{tokens}{'_gnorm' if gated else ''}", batch=64, tokens=tokens, slots=96, skipped=5,
                         gated_norm=gated, seed=tokens))


def test_decode_slots_grouped_heads_and_out_of_pool_index():
    _run(DecodeSlotsCase("slots_g3", batch=9, tokens=4, slots=12, skipped=1, out_of_pool=2,
                         hk=2, hv=6, seed=11))


def test_decode_slots_one_token_identity_slots_matches_gdn_decode():
    """tokens = 1 with no index is gdn_decode: same outputs and states, bit for bit."""
    import gated_deltanet_linear_08_gb300 as gdn
    x = make_decode_inputs(DecodeCase("id", batch=6, hk=2, hv=4, steps=1, gated_norm=True))
    dev = "cuda"
    st = {k: v.to(dev) for k, v in x["steps"][0].items()}
    A_log, dt = x["A_log"].to(dev), x["dt_bias"].to(dev)
    z, w = x["z"][0].to(dev), x["norm_w"].to(dev)
    S1, S2 = x["state"].to(dev), x["state"].to(dev)
    o1 = gdn.decode(st["q"], st["k"], st["v"], st["a"], st["b"], A_log, dt, S1, z=z, norm_w=w)
    o2 = gdn.decode_slots(*(st[n].unsqueeze(1) for n in ("q", "k", "v", "a", "b")), A_log, dt, S2,
                          z=z.unsqueeze(1), norm_w=w)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2[:, 0]) and torch.equal(S1, S2)
