"""gdn_prefill_noalloc: the prefill for callers that cannot allocate device
memory (hosts that hand a kernel only their own pre-registered buffers and
forbid allocation once running, or plain-C callers with no device
allocator).  Its scratch is the library's own fixed array, shared by every
call on the device, so this checks, through the C ABI, that back-to-back
calls on different problems give exactly (bit for bit) what the
workspace-taking gdn_prefill gives on the same inputs -- a stale read of the
shared array would show -- including a batch of 20 sequences (whose chunk
index also lives in the array) and the largest problem the array holds, and
that a problem one chunk larger is refused before any launch.

Collected last on purpose: if it fails, a run that stops at the first failure
has already run every other test.
"""
import ctypes

import pytest
import torch

from gated_deltanet_linear_08_gb300.inputs import PrefillCase, make_prefill_inputs
from parity_util import to_dev

pytestmark = pytest.mark.gpu

LIMIT = 64 << 20


def _both_paths(x):
    import gated_deltanet_linear_08_gb300 as gdn
    d = to_dev(x)
    args = (d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["cu_seqlens"])
    kw = dict(init_state=d["init_state"], z=d["z"], norm_w=d["norm_w"], eps=x["eps"])
    ref_out, ref_fin = gdn.prefill(*args, **kw)
    out, fin = gdn.prefill_noalloc(*args, **kw)
    torch.cuda.synchronize()
    assert gdn.check_device_status() == 0
    return ref_out, ref_fin, out, fin


def _equal(ref_out, ref_fin, out, fin):
    assert torch.equal(out, ref_out)
    assert torch.equal(fin, ref_fin)


def test_noalloc_matches_workspace_entry_point_twice():
    # different problems back to back through the one shared scratch array;
    # the second is the first again, after a larger one filled more of it
    first = make_prefill_inputs(PrefillCase("na1", seqlens=[100, 37, 64], hk=2, hv=4,
                                            init_state=True, gated_norm=True, seed=21))
    second = make_prefill_inputs(PrefillCase("na2", seqlens=[250], hk=2, hv=6,
                                             init_state=True, seed=22))
    for x in (first, second, first):
        _equal(*_both_paths(x))


def test_noalloc_many_sequences_use_the_chunk_index():
    # from 16 sequences on, the chunk index is built in the scratch array too
    lens = [0, 1, 63, 64, 65, 2, 17, 40, 5, 0] * 2
    x = make_prefill_inputs(PrefillCase("na_many", seqlens=lens, hk=2, hv=4, init_state=True,
                                        gated_norm=True, seed=23))
    _equal(*_both_paths(x))


def test_noalloc_largest_problem_fits_and_one_chunk_more_is_refused():
    import gated_deltanet_linear_08_gb300 as gdn
    from gated_deltanet_linear_08_gb300 import _binding as B
    # the largest single sequence at Hv = 32 whose workspace fits in the array
    T = max(t for t in range(64, 4096, 64) if B.workspace_bytes(1, t, 16, 32) <= LIMIT)
    assert B.workspace_bytes(1, T + 1, 16, 32) > LIMIT
    x = make_prefill_inputs(PrefillCase("na_limit", seqlens=[T], init_state=True, gated_norm=True, seed=24))
    _equal(*_both_paths(x))
    y = make_prefill_inputs(PrefillCase("na_over", seqlens=[T + 1], seed=25))
    d = to_dev(y)
    with pytest.raises(B.GdnError) as err:
        gdn.prefill_noalloc(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["cu_seqlens"])
    assert err.value.code == 6   # GDN_ERR_WORKSPACE


def test_noalloc_rejects_problems_beyond_its_scratch():
    from gated_deltanet_linear_08_gb300 import _binding as B
    lib = B.load()
    big = B.make_shape(1, 1 << 16, 16, 32)   # needs far more than 64 MiB
    assert B.workspace_bytes(1, 1 << 16, 16, 32) > LIMIT
    fake = 0x7f0000000000                    # never dereferenced: refused on the host
    code = lib.gdn_prefill_noalloc(ctypes.byref(big), fake, fake, fake, fake, fake, fake, fake,
                                   None, fake, None, None, 1e-6, fake, fake, None)
    assert code == 6   # GDN_ERR_WORKSPACE
