"""Serving-style integration of the path on the GPU (pegainfer page
"feat(qwen35): add SM120 FlashInfer GDN prefill candidate", Correctness:
chunked vs unchunked prefill with carried states; SGLang page "[Perf] Pack
the Qwen3.5 GDN input projection on CUDA", Accuracy Tests: mamba slots and
graph-captured decode).

  * prefill in 512-token pieces per call, several sequences at once, each
    call starting from the states the previous call returned, equals one
    call over the whole sequences bit for bit: piece boundaries are chunk
    boundaries, so every chunk sees the same tokens and the same fp32 state;
  * a decode loop over a slot pool captured in a CUDA graph and replayed
    equals the same calls made eagerly, bit for bit;
  * a captured prefill call equals the eager call;
  * prefill and decode on views into one packed buffer (one host copy per
    step in a serving loop) equal the calls on separate tensors.
"""
import numpy as np
import pytest
import torch

from gated_deltanet_linear_08_gb300.inputs import (DecodeSlotsCase, PrefillCase, make_decode_slots_inputs,
                                                   make_prefill_inputs)
from parity_util import to_dev

pytestmark = pytest.mark.gpu
PIECE = 512


def test_prefill_in_pieces_with_carried_states_matches_one_call():
    import gated_deltanet_linear_08_gb300 as gdn
    lens = [700, 1300, 64, 2000, 1]
    x = make_prefill_inputs(PrefillCase("pieces", seqlens=lens, hk=4, hv=8, init_state=True,
                                        gated_norm=True, seed=21))
    d = to_dev(x)
    full_out, full_fin = gdn.prefill(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                                     d["cu_seqlens"], init_state=d["init_state"], z=d["z"],
                                     norm_w=d["norm_w"], eps=x["eps"])
    starts = np.concatenate([[0], np.cumsum(lens)])
    states = d["init_state"].clone()
    out = torch.zeros_like(full_out)
    for i in range(max(lens) // PIECE + 1):
        live = [n for n in range(len(lens)) if lens[n] > PIECE * i]
        rows = [np.arange(starts[n] + PIECE * i, starts[n] + min(PIECE * (i + 1), lens[n])) for n in live]
        sel = torch.as_tensor(np.concatenate(rows), device="cuda")
        cu = torch.as_tensor(np.concatenate([[0], np.cumsum([len(r) for r in rows])]), dtype=torch.int32,
                             device="cuda")
        pick = lambda t: t.index_select(0, sel).contiguous()
        idx = torch.as_tensor(live, device="cuda")
        o, fin = gdn.prefill(pick(d["q"]), pick(d["k"]), pick(d["v"]), pick(d["a"]), pick(d["b"]),
                             d["A_log"], d["dt_bias"], cu, init_state=states.index_select(0, idx).contiguous(),
                             z=pick(d["z"]), norm_w=d["norm_w"], eps=x["eps"])
        out.index_copy_(0, sel, o)
        states.index_copy_(0, idx, fin)
    torch.cuda.synchronize()
    assert torch.equal(out, full_out)
    assert torch.equal(states, full_fin)
    assert gdn.check_device_status() == 0


@pytest.mark.parametrize("tokens", [1, 4])
def test_graph_captured_decode_loop_matches_eager(tokens):
    """A captured loop of slot-pool decode steps replays to the eager results
    bit for bit: one token per step (the single-token kernel) or a 4-token
    draft per step (the draft kernel)."""
    import gated_deltanet_linear_08_gb300 as gdn
    case = DecodeSlotsCase("graph", batch=16, tokens=tokens, slots=40, skipped=2, hk=4, hv=8, seed=5)
    steps = 12
    ys = [make_decode_slots_inputs(DecodeSlotsCase(case.name, batch=case.batch, tokens=tokens, slots=case.slots,
                                                   skipped=case.skipped, hk=case.hk, hv=case.hv, seed=100 + s))
          for s in range(steps)]
    base = make_decode_slots_inputs(case)
    toks = [{n: y[n].cuda() for n in ("q", "k", "v", "a", "b")} for y in ys]
    A_log, dt = base["A_log"].cuda(), base["dt_bias"].cuda()
    idx = base["state_idx"].cuda()
    outs_e = [torch.empty(case.batch, tokens, case.hv, 128, dtype=torch.bfloat16, device="cuda")
              for _ in range(steps)]
    outs_g = [torch.empty_like(o) for o in outs_e]

    def loop(pool, outs, stream=None):
        for s in range(steps):
            t = toks[s]
            gdn.decode_slots(t["q"], t["k"], t["v"], t["a"], t["b"], A_log, dt, pool, state_idx=idx,
                             out=outs[s], stream=stream)

    pool_e = base["pool"].cuda()
    loop(pool_e, outs_e)   # eager (also the warm-up before capture)
    pool_g = base["pool"].cuda()
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    pool_g0 = pool_g.clone()
    with torch.cuda.graph(graph, stream=stream):
        loop(pool_g, outs_g, stream=stream)
    pool_g.copy_(pool_g0)   # capture runs nothing; start the replay from the initial pool
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(pool_g, pool_e)
    assert all(torch.equal(a, b) for a, b in zip(outs_g, outs_e))
    assert gdn.check_device_status() == 0


def test_graph_captured_prefill_matches_eager():
    import gated_deltanet_linear_08_gb300 as gdn
    x = make_prefill_inputs(PrefillCase("gprefill", seqlens=[300, 65, 129], hk=2, hv=4, init_state=True,
                                        gated_norm=True, seed=8))
    d = to_dev(x)
    ws = gdn.alloc_workspace(3, d["q"].shape[0], 2, 4, "cuda")
    args = (d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["cu_seqlens"])
    kw = dict(init_state=d["init_state"], z=d["z"], norm_w=d["norm_w"], eps=x["eps"], workspace=ws)
    out_e, fin_e = gdn.prefill(*args, **kw)
    out_g, fin_g = torch.empty_like(out_e), torch.empty_like(fin_e)
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        gdn.prefill(*args, **kw, out=out_g, final_state=fin_g, stream=stream)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_g, out_e) and torch.equal(fin_g, fin_e)
    assert gdn.check_device_status() == 0


_FIRST_CALL_IN_CAPTURE = r"""
import sys, torch
sys.path.insert(0, {root!r})
import gated_deltanet_linear_08_gb300 as gdn
from gated_deltanet_linear_08_gb300.inputs import DecodeSlotsCase, make_decode_slots_inputs
x = make_decode_slots_inputs(DecodeSlotsCase("fresh", batch=8, tokens=4, slots=12, skipped=1, hk=2, hv=4, seed=9))
t = {{n: x[n].cuda() for n in ("q", "k", "v", "a", "b")}}
A_log, dt, idx = x["A_log"].cuda(), x["dt_bias"].cuda(), x["state_idx"].cuda()
pool_g, pool_e = x["pool"].cuda(), x["pool"].cuda()
out_g = torch.empty(8, 4, 4, 128, dtype=torch.bfloat16, device="cuda")
stream = torch.cuda.Stream()
graph = torch.cuda.CUDAGraph()
with torch.cuda.graph(graph, stream=stream):   # the library's first call of this process
    gdn.decode_slots(t["q"], t["k"], t["v"], t["a"], t["b"], A_log, dt, pool_g, state_idx=idx, out=out_g,
                     stream=stream)
graph.replay()
out_e = gdn.decode_slots(t["q"], t["k"], t["v"], t["a"], t["b"], A_log, dt, pool_e, state_idx=idx)
torch.cuda.synchronize()
assert torch.equal(out_g, out_e) and torch.equal(pool_g, pool_e)
assert gdn.check_device_status() == 0
print("ok")
"""


def test_first_draft_decode_call_inside_a_capture():
    """The draft kernel's one-time set-up (its shared-memory attribute and
    the resident-CTA count) runs inside a stream capture when the capture
    holds the process's first call; the replay still matches eager."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    res = subprocess.run([sys.executable, "-c", _FIRST_CALL_IN_CAPTURE.format(root=root)],
                         capture_output=True, text=True, timeout=300)
    assert res.returncode == 0 and res.stdout.strip().endswith("ok"), res.stdout + res.stderr


def test_calls_on_views_into_one_packed_buffer():
    """A serving loop that stages a step's inputs in one buffer (one copy
    per step) calls the library on typed views at 256-byte-aligned offsets
    of that buffer, and writes its results into views of another.  Prefill
    (gated norm) and decode through such views equal the same calls on
    separate tensors bit for bit."""
    import gated_deltanet_linear_08_gb300 as gdn
    from gated_deltanet_linear_08_gb300.inputs import DecodeCase, make_decode_inputs

    def pack(tensors):
        offs, n = [], 0
        for t in tensors:
            n = (n + 255) // 256 * 256
            offs.append(n)
            n += t.numel() * t.element_size()
        buf = torch.zeros((n + 255) // 256 * 256, dtype=torch.uint8, device="cuda")
        views = []
        for t, o in zip(tensors, offs):
            v = buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
            v.copy_(t)
            views.append(v)
        return buf, views

    x = make_prefill_inputs(PrefillCase("views", seqlens=[300, 77], hk=4, hv=8, init_state=True,
                                        gated_norm=True, seed=33))
    d = to_dev(x)
    keys = ("q", "k", "v", "a", "b", "z")
    _, pv = pack([d[k] for k in keys])
    p = dict(zip(keys, pv))
    T, hv, N = d["q"].shape[0], x["hv"], len(x["seqlens"])
    _, (out_v, fin_v) = pack([torch.zeros(T, hv, 128, dtype=torch.bfloat16, device="cuda"),
                              torch.zeros(N, hv, 128, 128, dtype=torch.float32, device="cuda")])
    gdn.prefill(p["q"], p["k"], p["v"], p["a"], p["b"], d["A_log"], d["dt_bias"], d["cu_seqlens"],
                init_state=d["init_state"], z=p["z"], norm_w=d["norm_w"], eps=x["eps"],
                out=out_v, final_state=fin_v)
    ref_out, ref_fin = gdn.prefill(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                                   d["cu_seqlens"], init_state=d["init_state"], z=d["z"],
                                   norm_w=d["norm_w"], eps=x["eps"])
    torch.cuda.synchronize()
    assert torch.equal(out_v, ref_out) and torch.equal(fin_v, ref_fin)

    y = make_decode_inputs(DecodeCase("views_dec", batch=24, hk=4, hv=8, steps=1, seed=34))
    st = {k: t.cuda() for k, t in y["steps"][0].items()}
    dkeys = ("q", "k", "v", "a", "b")
    _, dv = pack([st[k] for k in dkeys])
    s_views, s_ref = y["state"].cuda(), y["state"].cuda()
    A, dt = y["A_log"].cuda(), y["dt_bias"].cuda()
    o_v = gdn.decode(*dv, A, dt, s_views)
    o_r = gdn.decode(*(st[k] for k in dkeys), A, dt, s_ref)
    torch.cuda.synchronize()
    assert torch.equal(o_v, o_r) and torch.equal(s_views, s_ref)
    assert gdn.check_device_status() == 0
