"""GPU parity of the causal conv1d + SiLU fused ahead of the core (JevAny page
"Add opt-in fused Qwen3.5 inference kernels", Measurements: causal-conv1d is
one of the path's dependencies) against the fp64 oracle, on the seeded inputs
as drawn.

The conv output is rounded to bf16 on both sides; the kernels sum in fp32 and
the oracle in fp64, so an element whose exact value sits within the fp32
evaluation error of a bf16 rounding midpoint may round either way: both are
correct roundings, the conv's result is not unique there.  So each test
  1. takes the conv outputs the GPU produces: gdn_conv_prefill writes them
     out, and bitwise checks show that the prefill with the conv and the
     decode with its conv in registers compute exactly those values (their
     results equal the plain path's on them, bit for bit),
  2. checks that every one is a valid rounding of the exact fp64 value
     (parity_util.conv_check_rounding) and counts the ties rounded the other
     way,
  3. runs the oracle's core on those conv outputs and holds the GPU's core
     outputs and states to the usual bounds.
The carried conv states are raw inputs moved around, so they must match the
oracle's bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_08_gb300.inputs import (DecodeSlotsCase, PrefillCase, conv_channels, make_conv_inputs,
                                                   make_decode_slots_inputs, make_prefill_inputs, to_f64)
from parity_util import (DECODE_STATE_REL, assert_out_close, assert_state_close, conv_check_rounding, record,
                         to_dev)

pytestmark = pytest.mark.gpu


def _raw_rows(q, k, v):
    """q | k | v channels of each token as one [T, C] array (fp64)."""
    T = q.shape[0]
    return np.concatenate([to_f64(q).reshape(T, -1), to_f64(k).reshape(T, -1), to_f64(v).reshape(T, -1)], axis=1)


def _split(y, hk, hv, d=128):
    T = y.shape[0]
    return (y[:, :hk * d].reshape(T, hk, d), y[:, hk * d:2 * hk * d].reshape(T, hk, d),
            y[:, 2 * hk * d:].reshape(T, hv, d))


def _check_roundings(what, y_gpu, X, cu, w, states):
    """Validity of the GPU's conv outputs y_gpu [T, C] for raw rows X [T, C] of
    packed sequences cu (states[n]: [K-1, C] fp64 or None); records the count
    of ties rounded the other way."""
    flips = 0
    for n in range(len(cu) - 1):
        s, e = int(cu[n]), int(cu[n + 1])
        if e > s:
            flips += conv_check_rounding(y_gpu[s:e], X[s:e], w, states[n])
    record(what, "conv", dict(flips=flips, violations=0), "valid bf16 rounding of the exact value")
    return flips


def _gpu_prefill_conv(x, cv, in_place=False):
    """gdn.prefill with the conv; the conv outputs from gdn.conv_prefill, and
    the plain prefill on them, which must give the conv call's results bit for
    bit."""
    import gated_deltanet_linear_08_gb300 as gdn
    d = to_dev(x)
    hk, hv = x["q"].shape[1], x["v"].shape[1]
    w = cv["weight"].cuda()
    st = None if cv["state"] is None else cv["state"].cuda()
    y = gdn.conv_prefill(d["q"], d["k"], d["v"], d["cu_seqlens"], w, st)   # before the call rolls st in place
    out, fin, cs = gdn.prefill(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["cu_seqlens"],
                               init_state=d["init_state"], z=d["z"], norm_w=d["norm_w"], eps=x["eps"],
                               conv_weight=w, conv_state=st, conv_state_out=st if in_place else None)
    yq, yk, yv = (t.contiguous() for t in _split(y, hk, hv))
    out2, fin2 = gdn.prefill(yq, yk, yv, d["a"], d["b"], d["A_log"], d["dt_bias"], d["cu_seqlens"],
                             init_state=d["init_state"], z=d["z"], norm_w=d["norm_w"], eps=x["eps"])
    torch.cuda.synchronize()
    assert gdn.check_device_status() == 0
    assert torch.equal(out, out2) and torch.equal(fin, fin2), "the prefill's conv differs from gdn_conv_prefill's"
    return out, fin, cs, y.double().cpu().numpy()


def _check_prefill(case, width, with_state=True, in_place=False):
    x = make_prefill_inputs(case)
    cv = make_conv_inputs(conv_channels(case.hk, case.hv), width, len(x["seqlens"]), seed=case.seed,
                          state=with_state)
    out, fin, cs, y = _gpu_prefill_conv(x, cv, in_place=in_place)
    cu = x["cu_seqlens"].numpy()
    wf = to_f64(cv["weight"])
    states = [None if cv["state"] is None else to_f64(cv["state"][n]) for n in range(len(cu) - 1)]
    X = _raw_rows(x["q"], x["k"], x["v"])
    flips = _check_roundings(case.name + " conv outputs", y, X, cu, wf, states)
    # the oracle's core on the GPU's conv outputs
    qc, kc, vc = _split(y, case.hk, case.hv)
    f = {n: to_f64(x[n]) for n in ("a", "b", "A_log", "dt_bias", "init_state", "z", "norm_w")}
    ro, rs = oracle.prefill(cu, qc, kc, vc, f["a"], f["b"], f["A_log"], f["dt_bias"], f["init_state"], f["z"],
                            f["norm_w"], eps=x["eps"])
    so = assert_out_close(out.double().cpu().numpy(), ro, case.name + " out")
    ss = assert_state_close(fin.double().cpu().numpy(), rs, case.name + " state")
    # the carried conv states: the oracle's, bit for bit
    _, _, _, new = oracle.conv_inputs(cu, to_f64(x["q"]), to_f64(x["k"]), to_f64(x["v"]), wf,
                                      None if cv["state"] is None else to_f64(cv["state"]))
    assert np.array_equal(cs.double().cpu().numpy(), new), case.name + " conv state"
    print(case.name, "K", width, "ties rounded the other way", flips, "out", so, "state", ss)
    return x, cv, out, fin, cs


def test_prefill_conv_ragged_with_short_sequences():
    # lengths 1, 2 and 3 are shorter than or equal to K-1: their new conv state
    # keeps part of the old one
    _check_prefill(PrefillCase("conv_ragged", seqlens=[200, 64, 1, 2, 90, 130, 3], hk=2, hv=4, init_state=True,
                               gated_norm=True, seed=41), 4)


@pytest.mark.parametrize("width", [1, 2, 3, 4])
def test_prefill_conv_widths_grouped_heads(width):
    _check_prefill(PrefillCase(f"conv_w{width}", seqlens=[70, 2, 129], hk=2, hv=6, init_state=True, seed=42),
                   width)


def test_prefill_conv_zero_state_and_empty_sequences():
    _check_prefill(PrefillCase("conv_zero", seqlens=[0, 65, 0, 1, 128], hk=2, hv=4, seed=43), 4, with_state=False)
    x, cv, *_ = _check_prefill(PrefillCase("conv_empty", seqlens=[0, 65, 0, 1], hk=2, hv=4, seed=44), 4)


def test_prefill_conv_state_in_place_matches_out_of_place():
    case = PrefillCase("conv_inplace", seqlens=[150, 2, 64], hk=2, hv=4, init_state=True, seed=45)
    _, _, out_a, fin_a, cs_a = _check_prefill(case, 4)
    _, _, out_b, fin_b, cs_b = _check_prefill(case, 4, in_place=True)
    assert torch.equal(out_a, out_b) and torch.equal(fin_a, fin_b) and torch.equal(cs_a, cs_b)


def test_prefill_conv_T2048_workload():
    # the Qwen3.5-4B geometry at T=2048 with the gated RMSNorm, conv width 4
    _check_prefill(PrefillCase("conv_T2048", seqlens=[2048], gated_norm=True, init_state=True, seed=46), 4)


def test_prefill_conv_in_pieces_matches_one_call():
    """Two calls with the recurrent and conv states carried equal one call bit
    for bit: the piece boundary is a chunk boundary, and the carried conv
    state holds exactly the raw tokens the single call reads."""
    import gated_deltanet_linear_08_gb300 as gdn
    lens, cut = [300, 700], 256
    x = make_prefill_inputs(PrefillCase("conv_pieces", seqlens=lens, hk=2, hv=4, init_state=True, gated_norm=True,
                                        seed=47))
    cv = make_conv_inputs(conv_channels(2, 4), 4, 2, seed=47)
    d = to_dev(x)
    w, st = cv["weight"].cuda(), cv["state"].cuda()
    kw = dict(z=d["z"], norm_w=d["norm_w"], eps=x["eps"], conv_weight=w)
    full_out, full_fin, full_cs = gdn.prefill(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                                              d["cu_seqlens"], init_state=d["init_state"], conv_state=st, **kw)
    starts = [0, lens[0]]
    out = torch.empty_like(full_out)
    states, cstates = d["init_state"], st
    for lo, hi in ((0, cut), (cut, None)):
        rows = [torch.arange(s + lo, s + (l if hi is None else hi), device="cuda") for s, l in zip(starts, lens)]
        sel = torch.cat(rows)
        cu = torch.tensor([0, len(rows[0]), len(rows[0]) + len(rows[1])], dtype=torch.int32, device="cuda")
        pick = lambda t: t.index_select(0, sel).contiguous()
        o, states, cstates = gdn.prefill(pick(d["q"]), pick(d["k"]), pick(d["v"]), pick(d["a"]), pick(d["b"]),
                                         d["A_log"], d["dt_bias"], cu, init_state=states, conv_state=cstates,
                                         **dict(kw, z=pick(d["z"])))
        out.index_copy_(0, sel, o)
    torch.cuda.synchronize()
    assert torch.equal(out, full_out) and torch.equal(states, full_fin) and torch.equal(cstates, full_cs)
    assert gdn.check_device_status() == 0


def _gpu_conv_outputs(q, k, v, cu, weight, states):
    """The conv outputs gdn_conv_prefill produces for packed raw tokens q, k,
    v (bf16, [T, H, 128], CPU) of sequences cu with carried states [N, K-1,
    C]: bf16 [T, C] on the device."""
    import gated_deltanet_linear_08_gb300 as gdn
    dev = "cuda"
    y = gdn.conv_prefill(q.to(dev), k.to(dev), v.to(dev), torch.as_tensor(cu, dtype=torch.int32, device=dev),
                         weight.to(dev), states.to(dev) if states.numel() else None)
    torch.cuda.synchronize()
    return y


def _decode_conv(case, width, out_of_place=False):
    import gated_deltanet_linear_08_gb300 as gdn
    x = make_decode_slots_inputs(case)
    B, T, P = case.batch, case.tokens, case.slots
    hk, hv, d = case.hk, case.hv, case.d
    cv = make_conv_inputs(conv_channels(hk, hv), width, P, seed=case.seed)
    dev = "cuda"
    pool = x["pool"].to(dev)
    cpool = cv["state"].to(dev)
    cpool_in = cpool
    if out_of_place:
        # a second pool receives the rolled states; the first stays as it was
        fill = torch.full_like(cv["state"], 0.5)
        cpool = fill.to(dev)
    tok = {n: x[n].to(dev) for n in ("q", "k", "v", "a", "b")}
    zd = None if x["z"] is None else x["z"].to(dev)
    wd = None if x["norm_w"] is None else x["norm_w"].to(dev)
    idx_d = x["state_idx"].to(dev)
    out = gdn.decode_slots(tok["q"], tok["k"], tok["v"], tok["a"], tok["b"], x["A_log"].to(dev),
                           x["dt_bias"].to(dev), pool, state_idx=idx_d, z=zd, norm_w=wd, eps=x["eps"],
                           conv_weight=cv["weight"].to(dev), conv_state=cpool_in,
                           conv_state_out=cpool if out_of_place else None)
    bits = gdn.check_device_status()
    if out_of_place:
        assert torch.equal(cpool_in.cpu(), cv["state"])
    got_out, got_pool, got_cpool = out.double().cpu().numpy(), pool.cpu(), cpool.cpu()

    idx = x["state_idx"].numpy()
    live = np.nonzero((idx >= 0) & (idx < P))[0]
    dead = np.nonzero((idx < 0) | (idx >= P))[0]
    w = to_f64(cv["weight"])
    cst = to_f64(cv["state"])
    # 1. the conv outputs of the live sequences' drafts, from the prefill
    #    conv pass over the same raw tokens and carried states
    lv = torch.as_tensor(live)
    flat = lambda t: t[lv].flatten(0, 1).contiguous()
    cu = np.arange(0, len(live) * T + 1, T)
    y_dev = _gpu_conv_outputs(flat(x["q"]), flat(x["k"]), flat(x["v"]), cu, cv["weight"],
                              cv["state"][torch.as_tensor(idx[live].astype(np.int64))])
    y = y_dev.double().cpu().numpy()
    X = _raw_rows(flat(x["q"]), flat(x["k"]), flat(x["v"]))
    flips = _check_roundings(case.name + " conv outputs", y, X, cu, w, [cst[idx[n]] for n in live])
    # 2. decode computes exactly those conv outputs: the same decode without
    #    the conv, on them, gives the same outputs and states bit for bit
    yq, yk, yv = (t.reshape(len(live), T, *t.shape[1:]) for t in _split(y_dev, hk, hv))
    full = {n: tok[n].clone() for n in ("q", "k", "v")}
    lvd = lv.to(dev)
    full["q"][lvd], full["k"][lvd], full["v"][lvd] = yq, yk, yv
    pool2 = x["pool"].to(dev)
    out2 = gdn.decode_slots(full["q"], full["k"], full["v"], tok["a"], tok["b"], x["A_log"].to(dev),
                            x["dt_bias"].to(dev), pool2, state_idx=idx_d, z=zd, norm_w=wd, eps=x["eps"])
    torch.cuda.synchronize()
    gdn.check_device_status()
    assert torch.equal(out2[lvd], out[lvd]) and torch.equal(pool2, pool)
    # 3. the oracle: one decode step per token on those conv outputs
    yq, yk, yv = (np.asarray(t).reshape(len(live), T, *t.shape[1:]) for t in _split(y, hk, hv))
    S = np.ascontiguousarray(to_f64(x["pool"])[idx[live]])
    ref = np.zeros((len(live), T, hv, d))
    for t in range(T):
        ref[:, t] = oracle.decode_step(yq[:, t], yk[:, t], yv[:, t], to_f64(x["a"])[live, t],
                                       to_f64(x["b"])[live, t], to_f64(x["A_log"]), to_f64(x["dt_bias"]), S,
                                       z=None if x["z"] is None else to_f64(x["z"])[live, t],
                                       norm_w=to_f64(x["norm_w"]), eps=x["eps"])
    assert_out_close(got_out[live], ref, case.name + " out")
    Sg = got_pool[torch.as_tensor(idx[live].astype(np.int64))].double().numpy()
    rel = np.abs(Sg - S).max() / np.abs(S).max()
    record(case.name + " state", "state", dict(max_abs=float(rel), violations=int(rel > DECODE_STATE_REL)),
           f"max|dS|/max|S| <= {DECODE_STATE_REL:g}")
    assert rel <= DECODE_STATE_REL, rel
    assert np.all(got_out[dead] == 0)
    # 4. conv pool: named slots rolled exactly as the oracle rolls them,
    #    every other slot untouched
    for n in live:
        raw = np.concatenate([to_f64(x[m])[n].reshape(T, -1) for m in ("q", "k", "v")], axis=1)
        _, new = oracle.causal_conv_silu(raw, w, cst[idx[n]])
        assert np.array_equal(got_cpool[idx[n]].double().numpy(), new), idx[n]
    untouched = torch.as_tensor(np.setdiff1d(np.arange(P), idx[live]))
    assert torch.equal(got_cpool[untouched], (fill if out_of_place else cv["state"])[untouched])
    assert bits == (4 if case.out_of_pool else 0), bits
    print(case.name, "ties rounded the other way", flips)


@pytest.mark.parametrize("tokens", [1, 4])
def test_decode_conv_slots(tokens):
    _decode_conv(DecodeSlotsCase(f"conv_dec_T{tokens}", batch=48, tokens=tokens, slots=64, skipped=3,
                                 gated_norm=True, seed=50 + tokens), 4)


@pytest.mark.parametrize("tokens", [1, 2])
def test_decode_conv_into_a_second_pool(tokens):
    # the decode kernel writes the rolled states itself (no follow-up kernel)
    _decode_conv(DecodeSlotsCase(f"conv_dec_pp_T{tokens}", batch=40, tokens=tokens, slots=64, skipped=2,
                                 gated_norm=True, seed=56 + tokens), 4, out_of_place=True)
    _decode_conv(DecodeSlotsCase(f"conv_dec_pp_g3_T{tokens}", batch=9, tokens=tokens, slots=12, skipped=1,
                                 out_of_pool=1, hk=2, hv=6, seed=58 + tokens), 3, out_of_place=True)


@pytest.mark.parametrize("width", [1, 2, 3])
def test_decode_conv_widths_grouped_heads_out_of_pool(width):
    _decode_conv(DecodeSlotsCase(f"conv_dec_w{width}", batch=9, tokens=2, slots=12, skipped=1, out_of_pool=2,
                                 hk=2, hv=6, seed=60 + width), width)


def test_prefill_then_decode_with_conv_matches_one_prefill():
    """Serving order: prefill a prompt (recurrent and conv states out), then
    decode two tokens from those states.  The decoded outputs match the
    oracle's prefill over prompt + draft, run on the conv outputs the GPU
    produces for prompt + draft (checked as valid roundings)."""
    import gated_deltanet_linear_08_gb300 as gdn
    L, T, hk, hv = 133, 2, 2, 4
    x = make_prefill_inputs(PrefillCase("conv_serve", seqlens=[L + T, L + T], hk=hk, hv=hv, init_state=True,
                                        gated_norm=True, seed=48))
    cv = make_conv_inputs(conv_channels(hk, hv), 4, 2, seed=48)
    cu_full = x["cu_seqlens"].numpy()
    y_dev = _gpu_conv_outputs(x["q"], x["k"], x["v"], cu_full, cv["weight"], cv["state"])
    y = y_dev.double().cpu().numpy()
    _check_roundings("conv_serve conv outputs", y, _raw_rows(x["q"], x["k"], x["v"]), cu_full,
                     to_f64(cv["weight"]), [to_f64(cv["state"][n]) for n in range(2)])
    qc, kc, vc = _split(y, hk, hv)
    f = {n: to_f64(x[n]) for n in ("a", "b", "A_log", "dt_bias", "init_state", "z", "norm_w")}
    ro, _ = oracle.prefill(cu_full, qc, kc, vc, f["a"], f["b"], f["A_log"], f["dt_bias"], f["init_state"], f["z"],
                           f["norm_w"], eps=x["eps"])
    d = to_dev(x)
    w = cv["weight"].cuda()
    prompt = torch.cat([torch.arange(0, L), torch.arange(L + T, 2 * L + T)]).cuda()
    draft = torch.cat([torch.arange(L, L + T), torch.arange(2 * L + T, 2 * L + 2 * T)]).cuda()
    pick = lambda t, r: t.index_select(0, r).contiguous()
    cu = torch.tensor([0, L, 2 * L], dtype=torch.int32, device="cuda")
    _, fin, cst = gdn.prefill(*(pick(d[n], prompt) for n in ("q", "k", "v", "a", "b")), d["A_log"], d["dt_bias"],
                              cu, init_state=d["init_state"], z=pick(d["z"], prompt), norm_w=d["norm_w"],
                              eps=x["eps"], conv_weight=w, conv_state=cv["state"].cuda())
    dec = lambda t: pick(t, draft).unflatten(0, (2, T))
    out = gdn.decode_slots(*(dec(d[n]) for n in ("q", "k", "v", "a", "b")), d["A_log"], d["dt_bias"], fin,
                           z=dec(d["z"]), norm_w=d["norm_w"], eps=x["eps"], conv_weight=w, conv_state=cst)
    torch.cuda.synchronize()
    assert gdn.check_device_status() == 0
    assert_out_close(out.flatten(0, 1).double().cpu().numpy(), ro[draft.cpu().numpy()], "conv_serve draft out")


def test_graph_captured_decode_with_conv_matches_eager():
    import gated_deltanet_linear_08_gb300 as gdn
    case = DecodeSlotsCase("conv_graph", batch=8, tokens=1, slots=16, skipped=1, hk=2, hv=4, seed=70)
    x = make_decode_slots_inputs(case)
    cv = make_conv_inputs(conv_channels(2, 4), 4, 16, seed=70)
    t = {n: x[n].cuda() for n in ("q", "k", "v", "a", "b")}
    A_log, dt, idx, w = x["A_log"].cuda(), x["dt_bias"].cuda(), x["state_idx"].cuda(), cv["weight"].cuda()
    steps = 5

    def loop(pool, cpool, outs, stream=None):
        for s in range(steps):
            gdn.decode_slots(t["q"], t["k"], t["v"], t["a"], t["b"], A_log, dt, pool, state_idx=idx, out=outs[s],
                             stream=stream, conv_weight=w, conv_state=cpool)

    outs_e = [torch.empty(8, 1, 4, 128, dtype=torch.bfloat16, device="cuda") for _ in range(steps)]
    outs_g = [torch.empty_like(o) for o in outs_e]
    pool_e, cpool_e = x["pool"].cuda(), cv["state"].cuda()
    loop(pool_e, cpool_e, outs_e)
    pool_g, cpool_g = x["pool"].cuda(), cv["state"].cuda()
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        loop(pool_g, cpool_g, outs_g, stream=stream)
    pool_g.copy_(x["pool"].cuda())
    cpool_g.copy_(cv["state"].cuda())
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(pool_g, pool_e) and torch.equal(cpool_g, cpool_e)
    assert all(torch.equal(a, b) for a, b in zip(outs_g, outs_e))
    assert gdn.check_device_status() == 0


@pytest.mark.parametrize("out_of_place", [False, True])
def test_decode_conv_writes_nothing_past_the_pools_or_outputs(out_of_place):
    """Guard rows after the state pool, the conv-state pools and the output
    stay bit for bit as they were.  The out-of-pool index equals the pool
    size, so it names exactly the first guard row."""
    import gated_deltanet_linear_08_gb300 as gdn
    case = DecodeSlotsCase("conv_guard", batch=9, tokens=2, slots=12, skipped=1, out_of_pool=2, hk=2, hv=6,
                           seed=71)
    x = make_decode_slots_inputs(case)
    B, T, P, G = case.batch, case.tokens, case.slots, 2
    cv = make_conv_inputs(conv_channels(2, 6), 3, P + G, seed=71)
    dev = "cuda"
    pool = torch.cat([x["pool"], torch.full((G, 6, 128, 128), 3.0)]).to(dev)
    cin = cv["state"].to(dev)
    cout = torch.full_like(cin, 0.25) if out_of_place else cin
    out = torch.full((B + G, T, 6, 128), 5.0, dtype=torch.bfloat16, device=dev)
    guards = (pool[P:].clone(), cin[P:].clone(), cout[P:].clone(), out[B:].clone())
    gdn.decode_slots(*(x[n].to(dev) for n in ("q", "k", "v", "a", "b")), x["A_log"].to(dev), x["dt_bias"].to(dev),
                     pool[:P], state_idx=x["state_idx"].to(dev), out=out[:B], conv_weight=cv["weight"].to(dev),
                     conv_state=cin[:P], conv_state_out=cout[:P] if out_of_place else None)
    assert gdn.check_device_status() == 4   # the range bit for the out-of-pool indices
    for g, now in zip(guards, (pool[P:], cin[P:], cout[P:], out[B:])):
        assert torch.equal(g, now)
    dead = [i for i, s in enumerate(x["state_idx"].tolist()) if s < 0 or s >= P]
    assert bool((out[dead] == 0).all())


def test_prefill_conv_writes_nothing_past_the_states_or_outputs():
    import gated_deltanet_linear_08_gb300 as gdn
    x = make_prefill_inputs(PrefillCase("conv_guard_p", seqlens=[70, 2, 129], hk=2, hv=6, init_state=True,
                                        gated_norm=True, seed=72))
    N, T, G = 3, 201, 2
    cv = make_conv_inputs(conv_channels(2, 6), 4, N + G, seed=72)
    d = to_dev(x)
    cs_in = cv["state"].cuda()
    cs_out = torch.full_like(cs_in, 0.75)
    out = torch.full((T + G, 6, 128), 5.0, dtype=torch.bfloat16, device="cuda")
    fin = torch.full((N + G, 6, 128, 128), 9.0, device="cuda")
    guards = (cs_out[N:].clone(), out[T:].clone(), fin[N:].clone())
    gdn.prefill(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["cu_seqlens"],
                init_state=d["init_state"], z=d["z"], norm_w=d["norm_w"], eps=x["eps"], out=out[:T],
                final_state=fin[:N], conv_weight=cv["weight"].cuda(), conv_state=cs_in[:N], conv_state_out=cs_out[:N])
    assert gdn.check_device_status() == 0
    for g, now in zip(guards, (cs_out[N:], out[T:], fin[N:])):
        assert torch.equal(g, now)
