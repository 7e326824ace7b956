"""gdn_prefill_noalloc: the prefill for callers that cannot allocate device
memory (hosts that hand a kernel only their own pre-registered buffers, or
plain-C callers with no device allocator).  Its scratch is the library's own
fixed array, so this checks, through the C ABI, that two calls in a row give
what the workspace-taking gdn_prefill gives on the same inputs, and that a
problem larger than the array is refused before any launch.

Collected last on purpose: if it fails, a run that stops at the first failure
has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from gated_deltanet_linear_08_gb300.inputs import PrefillCase, make_prefill_inputs
from parity_util import OUT_MAX, OUT_MEAN, STATE_MAX, to_dev

pytestmark = pytest.mark.gpu


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


def _close(ref_out, ref_fin, out, fin):
    eo = (out.double() - ref_out.double()).abs()
    es = (fin.double() - ref_fin.double()).abs()
    assert torch.isfinite(out).all() and torch.isfinite(fin).all()
    assert eo.max().item() <= OUT_MAX and eo.mean().item() <= OUT_MEAN
    assert es.max().item() <= STATE_MAX


def test_noalloc_matches_workspace_entry_point_twice():
    # two different problems back to back through the one shared scratch array
    first = make_prefill_inputs(PrefillCase("na1", seqlens=[100, 37, 64], hk=2, hv=4,
                                            init_state=True, gated_norm=True, seed=21))
    second = make_prefill_inputs(PrefillCase("na2", seqlens=[250], hk=2, hv=6,
                                             init_state=True, seed=22))
    for x in (first, second):
        _close(*_both_paths(x))


def test_noalloc_rejects_problems_beyond_its_scratch():
    from gated_deltanet_linear_08_gb300 import _binding as B
    lib = B.load()
    big = B.make_shape(1, 1 << 16, 16, 32)   # needs far more than 64 MiB
    assert B.workspace_bytes(1, 1 << 16, 16, 32) > (64 << 20)
    fake = 0x7f0000000000                    # never dereferenced: refused on the host
    code = lib.gdn_prefill_noalloc(ctypes.byref(big), fake, fake, fake, fake, fake, fake, fake,
                                   None, fake, None, None, 1e-6, fake, fake, None)
    assert code == 6   # GDN_ERR_WORKSPACE
