"""GPU: the token inputs read in place from one packed projection output (SGLang
page "[Perf] Pack the Qwen3.5 GDN input projection on CUDA": a single GEMM on
the packed in_proj_qkvz and in_proj_ba weights writes each token's q, k, v,
z, b and a side by side).  The row order used here, q | k | v | z | b | a
(in_proj_qkvz rows, then in_proj_ba rows), is a reading: the page gives the
packed width but not the order, and the strided entry points accept any
order of head-contiguous blocks.  Results must equal the dense call bit for
bit: the same values reach the same arithmetic.
"""
import pytest
import torch

from gated_deltanet_linear_08_gb300.inputs import (DecodeSlotsCase, PrefillCase, make_decode_slots_inputs,
                                                   make_prefill_inputs)
from parity_util import to_dev

pytestmark = pytest.mark.gpu


def _pack(q, k, v, z, b, a):
    """One [tokens..., W] buffer holding q | k | v | z | b | a per token, and
    strided views of it shaped like the dense tensors."""
    lead = q.shape[:-2]
    parts = [q.flatten(-2), k.flatten(-2), v.flatten(-2), z.flatten(-2), b, a]
    W = sum(p.shape[-1] for p in parts)
    pad = (-W) % 8   # keep every block 16-byte aligned
    buf = torch.zeros(*lead, W + pad, dtype=torch.bfloat16, device=q.device)
    views, off = [], 0
    for p in parts:
        n = p.shape[-1]
        buf[..., off:off + n] = p
        views.append(buf[..., off:off + n])
        off += n
    qv = views[0].unflatten(-1, q.shape[-2:])
    kv = views[1].unflatten(-1, k.shape[-2:])
    vv = views[2].unflatten(-1, v.shape[-2:])
    zv = views[3].unflatten(-1, z.shape[-2:])
    return buf, qv, kv, vv, zv, views[4], views[5]


def test_prefill_reads_inputs_from_a_packed_projection():
    import gated_deltanet_linear_08_gb300 as gdn
    x = make_prefill_inputs(PrefillCase("packed", seqlens=[200, 64, 1, 90], hk=2, hv=4, init_state=True,
                                        gated_norm=True, seed=31))
    d = to_dev(x)
    ref_out, ref_fin = gdn.prefill(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                                   d["cu_seqlens"], init_state=d["init_state"], z=d["z"], norm_w=d["norm_w"],
                                   eps=x["eps"])
    buf, q, k, v, z, b, a = _pack(d["q"], d["k"], d["v"], d["z"], d["b"], d["a"])
    assert not q.is_contiguous() and q.stride(0) == buf.shape[-1]
    out, fin = gdn.prefill(q, k, v, a, b, d["A_log"], d["dt_bias"], d["cu_seqlens"], init_state=d["init_state"],
                           z=z, norm_w=d["norm_w"], eps=x["eps"])
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(fin, ref_fin)
    assert gdn.check_device_status() == 0


def test_single_chunk_prefill_reads_inputs_from_a_packed_projection():
    """A call of at most 64 tokens with no initial state, which prep finishes
    on its own (z read through the token and head strides), on packed
    inputs equals the dense call and the full path."""
    import gated_deltanet_linear_08_gb300 as gdn
    x = make_prefill_inputs(PrefillCase("packed_single", seqlens=[40, 0, 21], hk=2, hv=6, gated_norm=True,
                                        seed=35))
    d = to_dev(x)
    args = (d["A_log"], d["dt_bias"], d["cu_seqlens"])
    ref_out, ref_fin = gdn.prefill(d["q"], d["k"], d["v"], d["a"], d["b"], *args, z=d["z"], norm_w=d["norm_w"],
                                   eps=x["eps"])
    buf, q, k, v, z, b, a = _pack(d["q"], d["k"], d["v"], d["z"], d["b"], d["a"])
    out, fin = gdn.prefill(q, k, v, a, b, *args, z=z, norm_w=d["norm_w"], eps=x["eps"])
    zero = torch.zeros_like(ref_fin)
    full_out, full_fin = gdn.prefill(q, k, v, a, b, *args, init_state=zero, z=z, norm_w=d["norm_w"], eps=x["eps"])
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(fin, ref_fin)
    assert torch.equal(out, full_out) and torch.equal(fin, full_fin)
    assert gdn.check_device_status() == 0


def test_decode_reads_inputs_from_a_packed_projection():
    import gated_deltanet_linear_08_gb300 as gdn
    x = make_decode_slots_inputs(DecodeSlotsCase("packed_dec", batch=10, tokens=3, slots=16, skipped=1,
                                                 hk=2, hv=4, gated_norm=True, seed=32))
    dev = "cuda"
    t = {n: x[n].to(dev) for n in ("q", "k", "v", "a", "b", "z")}
    A_log, dt, idx, w = x["A_log"].to(dev), x["dt_bias"].to(dev), x["state_idx"].to(dev), x["norm_w"].to(dev)
    pool_ref, pool = x["pool"].to(dev), x["pool"].to(dev)
    ref = gdn.decode_slots(t["q"], t["k"], t["v"], t["a"], t["b"], A_log, dt, pool_ref, state_idx=idx,
                           z=t["z"], norm_w=w)
    buf, q, k, v, z, b, a = _pack(t["q"], t["k"], t["v"], t["z"], t["b"], t["a"])
    got = gdn.decode_slots(q, k, v, a, b, A_log, dt, pool, state_idx=idx, z=z, norm_w=w)
    torch.cuda.synchronize()
    assert torch.equal(got, ref) and torch.equal(pool, pool_ref)
    assert gdn.check_device_status() == 0


def test_conv_reads_inputs_from_a_packed_projection():
    """The serving order: one packed projection row per token, the causal conv
    over its q | k | v blocks, then the core.  Equal bit for bit to the same
    calls on dense copies, for prefill and for a slot-pool decode step."""
    import gated_deltanet_linear_08_gb300 as gdn
    from gated_deltanet_linear_08_gb300.inputs import conv_channels, make_conv_inputs
    x = make_prefill_inputs(PrefillCase("packed_conv", seqlens=[130, 2, 64], hk=2, hv=4, init_state=True,
                                        gated_norm=True, seed=33))
    d = to_dev(x)
    cv = make_conv_inputs(conv_channels(2, 4), 4, 3, seed=33)
    w, cs = cv["weight"].cuda(), cv["state"].cuda()
    common = dict(init_state=d["init_state"], norm_w=d["norm_w"], eps=x["eps"], conv_weight=w, conv_state=cs)
    ref = gdn.prefill(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["cu_seqlens"],
                      z=d["z"], **common)
    buf, q, k, v, z, b, a = _pack(d["q"], d["k"], d["v"], d["z"], d["b"], d["a"])
    got = gdn.prefill(q, k, v, a, b, d["A_log"], d["dt_bias"], d["cu_seqlens"], z=z, **common)
    torch.cuda.synchronize()
    assert all(torch.equal(g, r) for g, r in zip(got, ref))

    y = make_decode_slots_inputs(DecodeSlotsCase("packed_conv_dec", batch=6, tokens=2, slots=8, skipped=1,
                                                 hk=2, hv=4, gated_norm=True, seed=34))
    t = {n: y[n].cuda() for n in ("q", "k", "v", "a", "b", "z")}
    A_log, dt, idx, nw = y["A_log"].cuda(), y["dt_bias"].cuda(), y["state_idx"].cuda(), y["norm_w"].cuda()
    cvd = make_conv_inputs(conv_channels(2, 4), 4, 8, seed=34)
    wd = cvd["weight"].cuda()
    pool_r, pool_g = y["pool"].cuda(), y["pool"].cuda()
    cp_r, cp_g = cvd["state"].cuda(), cvd["state"].cuda()
    o_r = gdn.decode_slots(t["q"], t["k"], t["v"], t["a"], t["b"], A_log, dt, pool_r, state_idx=idx, z=t["z"],
                           norm_w=nw, conv_weight=wd, conv_state=cp_r)
    buf2, q2, k2, v2, z2, b2, a2 = _pack(t["q"], t["k"], t["v"], t["z"], t["b"], t["a"])
    o_g = gdn.decode_slots(q2, k2, v2, a2, b2, A_log, dt, pool_g, state_idx=idx, z=z2, norm_w=nw,
                           conv_weight=wd, conv_state=cp_g)
    torch.cuda.synchronize()
    assert torch.equal(o_g, o_r) and torch.equal(pool_g, pool_r) and torch.equal(cp_g, cp_r)
    assert gdn.check_device_status() == 0


def _pack_in_order(tensors: dict, order):
    """One [tokens..., W] buffer holding the named blocks in `order` per token,
    and strided views of it shaped like the dense tensors."""
    lead = tensors["q"].shape[:-2]
    flat = {n: (t.flatten(-2) if t.dim() == len(lead) + 2 else t) for n, t in tensors.items()}
    W = sum(flat[n].shape[-1] for n in order)
    buf = torch.zeros(*lead, W + (-W) % 8, dtype=torch.bfloat16, device=tensors["q"].device)
    views, off = {}, 0
    for n in order:
        m = flat[n].shape[-1]
        buf[..., off:off + m] = flat[n]
        views[n] = buf[..., off:off + m]
        if tensors[n].dim() == len(lead) + 2:
            views[n] = views[n].unflatten(-1, tensors[n].shape[-2:])
        off += m
        off += (-off) % 8 if n in ("a", "b") else 0   # keep the next 128-wide block 16-byte aligned
    return buf, views


ORDER = ("a", "z", "v", "b", "k", "q")   # not the q | k | v | z | b | a of the projection


def test_prefill_packed_hv48_against_the_oracle():
    """Packed inputs in a non-default block order, Hv = 48 (three value heads
    per k head): the outputs and final states follow the fp64 oracle."""
    import gated_deltanet_linear_08_gb300 as gdn
    from parity_util import assert_out_close, assert_state_close, oracle_prefill
    x = make_prefill_inputs(PrefillCase("packed_hv48", seqlens=[300, 1, 129, 64], hk=16, hv=48, init_state=True,
                                        gated_norm=True, seed=35))
    d = to_dev(x)
    buf, vw = _pack_in_order({n: d[n] for n in ("q", "k", "v", "z", "a", "b")}, ORDER)
    assert not vw["q"].is_contiguous() and vw["q"].stride(0) == buf.shape[-1]
    out, fin = gdn.prefill(vw["q"], vw["k"], vw["v"], vw["a"], vw["b"], d["A_log"], d["dt_bias"], d["cu_seqlens"],
                           init_state=d["init_state"], z=vw["z"], norm_w=d["norm_w"], eps=x["eps"])
    torch.cuda.synchronize()
    assert gdn.check_device_status() == 0
    ro, rs = oracle_prefill(x)
    assert_out_close(out.double().cpu().numpy(), ro, "packed_hv48 prefill out")
    assert_state_close(fin.double().cpu().numpy(), rs, "packed_hv48 prefill state")


def test_decode_packed_hv48_against_the_oracle():
    """Slot-pool decode of 3 draft tokens with packed inputs in a non-default
    block order at Hv = 48: outputs and states follow the fp64 oracle token
    by token."""
    import numpy as np

    import gated_deltanet_linear_08_gb300 as gdn
    import oracle
    from gated_deltanet_linear_08_gb300.inputs import to_f64
    from parity_util import DECODE_STATE_REL, assert_out_close, record
    case = DecodeSlotsCase("packed_dec_hv48", batch=24, tokens=3, slots=32, skipped=2, hk=16, hv=48,
                           gated_norm=True, seed=36)
    x = make_decode_slots_inputs(case)
    dev = "cuda"
    t = {n: x[n].to(dev) for n in ("q", "k", "v", "a", "b", "z")}
    pool = x["pool"].to(dev)
    buf, vw = _pack_in_order(t, ORDER)
    out = gdn.decode_slots(vw["q"], vw["k"], vw["v"], vw["a"], vw["b"], x["A_log"].to(dev), x["dt_bias"].to(dev),
                           pool, state_idx=x["state_idx"].to(dev), z=vw["z"], norm_w=x["norm_w"].to(dev),
                           eps=x["eps"])
    torch.cuda.synchronize()
    assert gdn.check_device_status() == 0
    idx = x["state_idx"].numpy()
    live = np.nonzero(idx >= 0)[0]
    S = np.ascontiguousarray(to_f64(x["pool"])[idx[live]])
    T = case.tokens
    ref = np.zeros((len(live), T, case.hv, 128))
    for s in range(T):
        ref[:, s] = oracle.decode_step(*(to_f64(x[n])[live, s] for n in ("q", "k", "v", "a", "b")),
                                       to_f64(x["A_log"]), to_f64(x["dt_bias"]), S, z=to_f64(x["z"])[live, s],
                                       norm_w=to_f64(x["norm_w"]), eps=x["eps"])
    got = out.double().cpu().numpy()
    assert_out_close(got[live], ref, "packed_dec_hv48 out")
    assert np.all(got[idx < 0] == 0)
    Sg = pool.cpu()[torch.as_tensor(idx[live].astype(np.int64))].double().numpy()
    rel = float(np.abs(Sg - S).max() / np.abs(S).max())
    record("packed_dec_hv48 state", "state", dict(max_abs=rel, violations=int(rel > DECODE_STATE_REL)),
           f"max|dS|/max|S| <= {DECODE_STATE_REL:g}")
    assert rel <= DECODE_STATE_REL
