"""GPU parity of gdn_prefill against the fp64 oracle.

Covers the four prefill workloads (T=64; 8x128 packed with initial states;
T=2048 with the gated-RMSNorm epilogue, also as 2x1024 with the state
carried; 16 varlen sequences at Hv=48), the chunk boundaries the pegainfer
page tests ("feat(qwen35): add SM120 FlashInfer GDN prefill candidate",
Correctness: T = 1, 2, 63, 64, 65, 127, 128; chunked vs unchunked prefill),
grouped heads, empty sequences, in-place state, weak and pure decay, long
sequences (16,384 tokens; 8,192 with weak decay), run-to-run determinism,
and the single-chunk calls that prep finishes on its own.
"""
import math

import numpy as np
import pytest
import torch

from gated_deltanet_linear_08_gb300.inputs import (CASE_8x128, CASE_T64, CASE_T2048,
                                                   CASE_VARLEN48, PrefillCase,
                                                   make_prefill_inputs)
from parity_util import (assert_out_close, assert_state_close, gpu_prefill, oracle_prefill,
                         out_stats, state_stats)

pytestmark = pytest.mark.gpu


def _check(case, in_place=False, scale_state=False):
    x = make_prefill_inputs(case)
    ro, rs = oracle_prefill(x)
    go, gs = gpu_prefill(x, in_place=in_place)
    so = assert_out_close(go, ro, case.name + " out")
    ss = assert_state_close(gs, rs, case.name + " state", scale_with_ref=scale_state)
    print(case.name, "out", so, "state", ss)
    return x, go, gs


@pytest.mark.parametrize("case", [CASE_T64, CASE_8x128, CASE_T2048, CASE_VARLEN48],
                         ids=lambda c: c.name)
def test_prefill_workloads(case):
    _check(case)


@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 127, 128])
def test_prefill_chunk_boundaries(T):
    _check(PrefillCase(f"T{T}", seqlens=[T], init_state=True, seed=T))


def test_prefill_grouped_heads_ratio3_and_ragged():
    _check(PrefillCase("g3", seqlens=[70, 1, 130, 64], hk=2, hv=6, init_state=True, seed=3))


def test_prefill_empty_sequences():
    x, go, gs = _check(PrefillCase("empty", seqlens=[0, 5, 0, 64, 0], hk=2, hv=4,
                                   init_state=True, seed=4))
    init = x["init_state"].double().numpy()
    for n in (0, 2, 4):
        assert np.array_equal(gs[n], init[n])


def test_prefill_in_place_state():
    _check(PrefillCase("inplace", seqlens=[100, 28], hk=2, hv=4, init_state=True, seed=5),
           in_place=True)


def test_prefill_weak_decay_carries_state():
    _check(PrefillCase("weak", seqlens=[700], hk=2, hv=4, init_state=True, seed=6,
                       a_log_const=math.log(0.01)), scale_state=True)


def test_prefill_long_sequence_16k_tokens():
    """One 16,384-token sequence (256 chunks per chain, eight times the
    T = 2048 workload's) with initial states and the gated norm: the scan's
    stage ring streams a long chain, the output kernel walks ~55 units per CTA."""
    _check(PrefillCase("T16384_gnorm", seqlens=[16384], init_state=True, gated_norm=True, seed=16))


def test_prefill_long_weak_decay_carries_state():
    """8,192 tokens with weak decay: the state carries across many chunks, so
    the fp16 operand roundings of 128 chunk steps accumulate in it."""
    _check(PrefillCase("weak_T8192", seqlens=[8192], hk=2, hv=4, init_state=True, seed=17,
                       a_log_const=math.log(0.01)), scale_state=True)


def test_prefill_pure_decay():
    """b -> -inf gives beta = 0: the state only decays (e^{sum g} S0)."""
    _check(PrefillCase("decay", seqlens=[150], hk=2, hv=4, init_state=True, seed=7,
                       a_log_const=math.log(0.02), b_const=-1e4))


def test_prefill_gated_norm_small():
    _check(PrefillCase("gn", seqlens=[65, 130], hk=2, hv=4, init_state=True, gated_norm=True,
                       seed=8))


@pytest.mark.parametrize("gated", [False, True])
def test_prefill_2x1024_carried_state_matches_single_call(gated):
    """T=2048 in one call vs two 1024-token calls with the state carried: chunk
    boundaries coincide, so the results are bitwise equal."""
    import gated_deltanet_linear_08_gb300 as gdn
    x = make_prefill_inputs(PrefillCase("c", seqlens=[2048], gated_norm=gated, init_state=True,
                                        seed=9))
    dev = "cuda"
    d = {k: (None if x[k] is None else x[k].to(dev)) for k in
         ("q", "k", "v", "a", "b", "A_log", "dt_bias", "init_state", "z", "norm_w")}
    cu = x["cu_seqlens"].to(dev)
    out1, fin1 = gdn.prefill(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], cu,
                             init_state=d["init_state"], z=d["z"], norm_w=d["norm_w"], eps=x["eps"])
    half = torch.tensor([0, 1024], dtype=torch.int32, device=dev)
    sl = lambda t, lo, hi: None if t is None else t[lo:hi].contiguous()
    oa, fa = gdn.prefill(sl(d["q"], 0, 1024), sl(d["k"], 0, 1024), sl(d["v"], 0, 1024),
                         sl(d["a"], 0, 1024), sl(d["b"], 0, 1024), d["A_log"], d["dt_bias"], half,
                         init_state=d["init_state"], z=sl(d["z"], 0, 1024), norm_w=d["norm_w"],
                         eps=x["eps"])
    ob, fb = gdn.prefill(sl(d["q"], 1024, 2048), sl(d["k"], 1024, 2048), sl(d["v"], 1024, 2048),
                         sl(d["a"], 1024, 2048), sl(d["b"], 1024, 2048), d["A_log"], d["dt_bias"],
                         half, init_state=fa, z=sl(d["z"], 1024, 2048), norm_w=d["norm_w"],
                         eps=x["eps"])
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([oa, ob]), out1)
    assert torch.equal(fb, fin1)


LONG_AMONG_TINY = [700] + [1] * 10   # an 11-chunk chain among single-token ones


@pytest.mark.parametrize("lens", [[300, 17], [70, 1, 64, 129, 5, 300, 2, 63] * 3, LONG_AMONG_TINY],
                         ids=["two_long", "24_short", "long_among_tiny"])
def test_prefill_deterministic_and_stream(lens):
    """Repeated calls, and a call on a side stream, agree bit for bit: every
    record a kernel writes is complete before the kernel that reads it, and
    no stage is refilled under the reads of the chunk before (24 short
    sequences also take the chunk index)."""
    x = make_prefill_inputs(PrefillCase("det", seqlens=lens, hk=2, hv=4, init_state=True,
                                        gated_norm=True, seed=10))
    o1, s1 = gpu_prefill(x)
    for _ in range(8):
        o3, s3 = gpu_prefill(x)
        assert np.array_equal(o1, o3) and np.array_equal(s1, s3)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        o2, s2 = gpu_prefill(x, stream=st)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)


def test_prefill_long_chain_among_tiny_ones():
    """A long sequence among single-token ones, 11 chunks on one chain: each
    chunk's S record, and so the early rows of every chunk's outputs, follows
    the oracle."""
    _check(PrefillCase("long_tiny", seqlens=LONG_AMONG_TINY, hk=2, hv=4, init_state=True,
                       gated_norm=True, seed=14))


def _sub_batch(x, first, last):
    """Sequences first .. last-1 of a packed batch as a batch of their own."""
    cu = x["cu_seqlens"]
    s, e = int(cu[first]), int(cu[last])
    y = dict(x)
    y["seqlens"] = x["seqlens"][first:last]
    y["cu_seqlens"] = (cu[first:last + 1] - s).to(torch.int32)
    for key in ("q", "k", "v", "a", "b", "z"):
        y[key] = None if x[key] is None else x[key][s:e].contiguous()
    y["init_state"] = None if x["init_state"] is None else x["init_state"][first:last].contiguous()
    return y, s, e


def test_prefill_units_past_the_output_kernels_unit_list():
    """640 sequences of 128 tokens at Hv=32: 40960 (chunk, head) units, about
    270 per output-kernel CTA, so each CTA locates its units past the first
    256 on the way instead of from the list it builds up front.  Sequences
    at both ends of the batch (the last ones are all past the list) follow
    the oracle run on them alone."""
    x = make_prefill_inputs(PrefillCase("units", seqlens=[128] * 640, hk=16, hv=32, gated_norm=True,
                                        seed=21))
    go, gs = gpu_prefill(x)
    for first, last in ((0, 2), (636, 640)):
        sub, s, e = _sub_batch(x, first, last)
        ro, rs = oracle_prefill(sub)
        assert_out_close(go[s:e], ro, f"units {first}-{last} out")
        assert_state_close(gs[first:last], rs, f"units {first}-{last} state")


def test_prefill_many_sequences_use_the_chunk_index():
    """40 packed sequences (empty, single-token, boundary and multi-chunk
    lengths): from 16 sequences on, the kernels find their chunks through the
    chunk index instead of walking cu_seqlens."""
    lens = [0, 1, 63, 64, 65, 130, 2, 0, 200, 17] * 4
    _check(PrefillCase("many40", seqlens=lens, hk=2, hv=4, init_state=True, gated_norm=True, seed=12))


def test_prefill_index_path_equals_walk_path():
    """24 sequences in one call (chunk index) equal the same sequences in two
    calls of 12 (walking cu_seqlens), bit for bit."""
    import gated_deltanet_linear_08_gb300 as gdn
    lens = [70, 1, 0, 64, 129, 5, 300, 2, 63, 65, 0, 40] * 2
    x = make_prefill_inputs(PrefillCase("idxwalk", seqlens=lens, hk=2, hv=4, init_state=True, gated_norm=True,
                                        seed=13))
    from parity_util import to_dev
    d = to_dev(x)
    kw = dict(z=d["z"], norm_w=d["norm_w"], eps=x["eps"])
    out, fin = gdn.prefill(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["cu_seqlens"],
                           init_state=d["init_state"], **kw)
    cu = x["cu_seqlens"].tolist()
    half = cu[12]
    for lo, hi, tl, th in ((0, 12, 0, half), (12, 24, half, cu[24])):
        sl = slice(tl, th)
        cu_h = torch.tensor([c - tl for c in cu[lo:hi + 1]], dtype=torch.int32, device="cuda")
        o, f = gdn.prefill(d["q"][sl].contiguous(), d["k"][sl].contiguous(), d["v"][sl].contiguous(),
                           d["a"][sl].contiguous(), d["b"][sl].contiguous(), d["A_log"], d["dt_bias"], cu_h,
                           init_state=d["init_state"][lo:hi].contiguous(), z=d["z"][sl].contiguous(),
                           norm_w=d["norm_w"], eps=x["eps"])
        torch.cuda.synchronize()
        assert torch.equal(o, out[sl]) and torch.equal(f, fin[lo:hi])
    assert gdn.check_device_status() == 0


@pytest.mark.parametrize("nseq", [3, 20])
def test_prefill_malformed_seqlens_are_flagged_and_skipped(nseq):
    """A sequence whose end lies past the packed tokens is treated as empty
    (its final state is its initial state) and sets the status bit; the others
    are computed as usual.  Both the walk (3 sequences) and the chunk index
    (20) are covered."""
    import gated_deltanet_linear_08_gb300 as gdn
    lens = [64, 70, 9, 130][: nseq - 1] if nseq < 5 else ([64, 70, 9, 130] * 5)[: nseq - 1]
    x = make_prefill_inputs(PrefillCase(f"bad{nseq}", seqlens=lens, hk=2, hv=4, init_state=True, seed=14))
    T = x["q"].shape[0]
    from parity_util import to_dev
    d = to_dev(x)
    N = len(lens) + 1
    cu = torch.tensor(x["cu_seqlens"].tolist() + [T + 7], dtype=torch.int32, device="cuda")   # past the end
    init = torch.cat([d["init_state"], torch.full((1, 4, 128, 128), 0.25, device="cuda")])
    out, fin = gdn.prefill(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], cu, init_state=init)
    assert gdn.check_device_status() == 2
    ro, rs = oracle_prefill(x)
    assert_out_close(out.double().cpu().numpy(), ro, f"bad{nseq} out")
    assert_state_close(fin[:N - 1].double().cpu().numpy(), rs, f"bad{nseq} state")
    assert torch.equal(fin[N - 1], init[N - 1])


def test_prefill_more_chains_than_scan_ctas():
    """48 sequences at Hv=32: 6144 chains (sequence, head, value slice), far
    more than fit on the GPU at once, so every scan CTA runs about 40 chains
    in turn (the stages and S buffers carried over chain boundaries, the next
    chain's initial state loaded during the current one).  Sequences at both
    ends of the batch follow the oracle run on them alone, and a repeat of
    the call agrees bit for bit."""
    lens = [1, 63, 64, 65, 130, 200] * 8
    x = make_prefill_inputs(PrefillCase("chains", seqlens=lens, hk=16, hv=32, init_state=True, gated_norm=True,
                                        seed=22))
    go, gs = gpu_prefill(x)
    go2, gs2 = gpu_prefill(x)
    assert np.array_equal(go, go2) and np.array_equal(gs, gs2)
    for first, last in ((0, 3), (45, 48)):
        sub, s, e = _sub_batch(x, first, last)
        ro, rs = oracle_prefill(sub)
        assert_out_close(go[s:e], ro, f"chains {first}-{last} out")
        assert_state_close(gs[first:last], rs, f"chains {first}-{last} state")


@pytest.mark.parametrize("lens,gated", [([64], True), ([1], False), ([63], True), ([30, 0, 34], False),
                                        ([3, 0, 0, 5, 1, 0, 7, 2, 0, 9, 4, 0, 6, 1, 0, 8, 3, 0, 2, 5], True)],
                         ids=["T64_gnorm", "T1", "T63_gnorm", "three_one_empty", "twenty_with_index"])
def test_prefill_single_chunk_call_equals_the_scan_path(lens, gated):
    """A call of 64 tokens or fewer with no initial state is finished inside
    prep (no scan or output kernel).  It equals the same call with an
    explicit all-zero initial state, which runs every kernel, bit for bit
    (outputs and final states, empty sequences included), and the oracle."""
    import gated_deltanet_linear_08_gb300 as gdn
    x = make_prefill_inputs(PrefillCase("single", seqlens=lens, hk=16, hv=32, gated_norm=gated, seed=41))
    from parity_util import to_dev
    d = to_dev(x)
    N = len(lens)
    args = (d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["cu_seqlens"])
    kw = dict(z=d["z"], norm_w=d["norm_w"], eps=x["eps"])
    o1, s1 = gdn.prefill(*args, **kw)
    zero = torch.zeros(N, 32, 128, 128, dtype=torch.float32, device="cuda")
    o2, s2 = gdn.prefill(*args, init_state=zero, **kw)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
    assert torch.equal(s1, s2)
    for n in range(N):
        if lens[n] == 0:
            assert int(torch.count_nonzero(s1[n])) == 0
    assert gdn.check_device_status() == 0
    ro, rs = oracle_prefill(x)
    assert_out_close(o1.double().cpu().numpy(), ro, "single out")
    assert_state_close(s1.double().cpu().numpy(), rs, "single state")
