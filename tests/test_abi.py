"""Host-side checks of the C ABI (no GPU): the library builds and loads, exports
every function include/gdn.h declares, and rejects bad arguments with the
documented status codes before any CUDA call (pegainfer page, maintainer
review: a stable C ABI, unsupported shapes handled explicitly).

The pointers passed here are fake integers; every case returns during host
validation, before anything could dereference them or touch a device.
"""
import ctypes
import os
import re

import pytest

from gated_deltanet_linear_08_gb300 import _binding as B
from gated_deltanet_linear_08_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return B.load()


def _declared_functions():
    with open(os.path.join(ROOT, "include", "gdn.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert set(names) == set(B.EXPORTED), names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code, name in B.STATUS_NAMES.items():
        assert B.status_string(code).startswith(name)
    assert B.status_string(99) == "GDN_ERR_UNKNOWN"


def test_workspace_bytes_formula(lib):
    # one 137 KiB record per (chunk, v head), chunks <= ceil(T/64) + N, then the
    # chunk index (int32 [N+1], 1 KiB aligned)
    assert B.workspace_bytes(1, 2048, 16, 32) == (32 + 1) * 32 * 140288 + 1024
    assert B.workspace_bytes(8, 1024, 16, 32) == (16 + 8) * 32 * 140288 + 1024
    assert B.workspace_bytes(300, 1024, 16, 32) == (16 + 300) * 32 * 140288 + 2048
    assert B.workspace_bytes(3, 0, 16, 32) == 0
    s = B.make_shape(1, 64, 16, 32, dk=64)
    assert lib.gdn_prefill_workspace_bytes(ctypes.byref(s)) == 0   # unsupported -> 0


FAKE = 0x7f0000000000   # 1024-byte aligned, never dereferenced


def _prefill(lib, shape, **kw):
    args = dict(q=FAKE, k=FAKE + 0x10000000, v=FAKE + 0x20000000, a=FAKE + 0x30000000,
                b=FAKE + 0x40000000, A_log=FAKE + 0x50000000, dt_bias=FAKE + 0x60000000,
                init=None, cu=FAKE + 0x70000000, z=None, w=None, eps=1e-6,
                out=FAKE + 0x80000000, fin=FAKE + 0x90000000, ws=FAKE + 0xA0000000,
                ws_bytes=1 << 40)
    args.update(kw)
    return lib.gdn_prefill(ctypes.byref(shape) if shape is not None else None, args["q"],
                           args["k"], args["v"], args["a"], args["b"], args["A_log"],
                           args["dt_bias"], args["init"], args["cu"], args["z"], args["w"],
                           args["eps"], args["out"], args["fin"], args["ws"], args["ws_bytes"],
                           None)


def test_prefill_rejects_bad_arguments(lib):
    ok = B.make_shape(1, 64, 16, 32)
    assert _prefill(lib, None) == 1
    assert _prefill(lib, B.make_shape(1, 64, 16, 32, dk=64)) == 2
    assert _prefill(lib, B.make_shape(1, 64, 16, 32, dv=256)) == 2
    assert _prefill(lib, B.make_shape(1, 64, 16, 32, hq=32)) == 2
    assert _prefill(lib, B.make_shape(1, 64, 16, 40)) == 2
    assert _prefill(lib, B.make_shape(-1, 64, 16, 32)) == 1
    assert _prefill(lib, ok, q=None) == 1
    assert _prefill(lib, ok, cu=None) == 1
    assert _prefill(lib, ok, z=FAKE + 0xB0000000) == 1          # z without norm_w
    assert _prefill(lib, ok, eps=-1.0) == 1
    assert _prefill(lib, ok, q=FAKE + 8) == 3                   # misaligned bf16 tensor
    assert _prefill(lib, ok, ws=FAKE + 0xA0000000 + 512) == 3   # workspace not 1024-aligned
    assert _prefill(lib, ok, ws=None) == 6
    assert _prefill(lib, ok, ws_bytes=1000) == 6
    assert _prefill(lib, ok, out=FAKE + 0x100) == 1             # out overlaps q
    assert _prefill(lib, ok, init=FAKE + 0x90000000 + 4096) == 1  # partial state overlap
    assert _prefill(lib, B.make_shape(0, 5, 16, 32)) == 1       # tokens without sequences
    assert _prefill(lib, B.make_shape(0, 0, 16, 32)) == 0       # empty problem: no-op


def test_decode_rejects_bad_arguments(lib):
    def dec(shape, **kw):
        a = dict(q=FAKE, k=FAKE + 0x10000000, v=FAKE + 0x20000000, a=FAKE + 0x30000000,
                 b=FAKE + 0x40000000, A_log=FAKE + 0x50000000, dt=FAKE + 0x60000000,
                 state=FAKE + 0x70000000, z=None, w=None, eps=1e-6, out=FAKE + 0x90000000)
        a.update(kw)
        return lib.gdn_decode(ctypes.byref(shape), a["q"], a["k"], a["v"], a["a"], a["b"],
                              a["A_log"], a["dt"], a["state"], a["z"], a["w"], a["eps"],
                              a["out"], None)
    assert dec(B.make_shape(4, 5, 16, 32)) == 1                 # total_tokens != batch
    assert dec(B.make_shape(4, 4, 16, 32, dk=96)) == 2
    assert dec(B.make_shape(4, 4, 16, 32), state=None) == 1
    assert dec(B.make_shape(4, 4, 16, 32), v=FAKE + 0x20000000 + 2) == 3
    assert dec(B.make_shape(4, 4, 16, 32), out=FAKE + 0x70000000) == 1   # out overlaps state
    assert dec(B.make_shape(0, 0, 16, 32)) == 0


def test_decode_slots_rejects_bad_arguments(lib):
    # host-side validation only: every call here fails before any launch
    def dec(shape, tokens=2, slots=8, **kw):
        a = dict(q=FAKE, k=FAKE + 0x10000000, v=FAKE + 0x20000000, a=FAKE + 0x30000000,
                 b=FAKE + 0x40000000, A_log=FAKE + 0x50000000, dt=FAKE + 0x60000000,
                 state=FAKE + 0x70000000, idx=FAKE + 0x80000000, z=None, w=None, eps=1e-6,
                 out=FAKE + 0x90000000)
        a.update(kw)
        return lib.gdn_decode_slots(ctypes.byref(shape), tokens, slots, a["q"], a["k"], a["v"], a["a"],
                                    a["b"], a["A_log"], a["dt"], a["state"], a["idx"], a["z"], a["w"],
                                    a["eps"], a["out"], None)
    assert dec(B.make_shape(4, 8, 16, 32), tokens=0) == 1         # tokens outside 1..8
    assert dec(B.make_shape(4, 36, 16, 32), tokens=9) == 1
    assert dec(B.make_shape(4, 7, 16, 32)) == 1                   # total_tokens != B * tokens
    assert dec(B.make_shape(4, 8, 16, 32), slots=-1) == 1
    assert dec(B.make_shape(4, 8, 16, 32), slots=3, idx=None) == 1   # identity slots need P >= B
    assert dec(B.make_shape(4, 8, 16, 32), idx=FAKE + 0x80000000 + 2) == 3   # index not 4-byte aligned
    assert dec(B.make_shape(4, 8, 16, 32), out=FAKE + 0x70000000) == 1       # out overlaps the pool
    assert dec(B.make_shape(4, 8, 16, 32, dv=64)) == 2
    assert dec(B.make_shape(0, 0, 16, 32)) == 0                   # empty batch: no-op


def test_strided_entry_points_reject_bad_strides(lib):
    # host-side validation only: every call here fails before any launch
    def strides(**over):
        base = dict(q=(16 * 128, 128), k=(16 * 128, 128), v=(32 * 128, 128), z=(32 * 128, 128),
                    a=(32, 1), b=(32, 1))
        base.update(over)
        return B.Strides(*(B.Stride(*base[n]) for n in ("q", "k", "v", "z", "a", "b")))

    def pre(st):
        return lib.gdn_prefill_strided(ctypes.byref(B.make_shape(1, 64, 16, 32)), ctypes.byref(st), FAKE,
                                       FAKE + 0x10000000, FAKE + 0x20000000, FAKE + 0x30000000,
                                       FAKE + 0x40000000, FAKE + 0x50000000, FAKE + 0x60000000, None,
                                       FAKE + 0x80000000, None, None, 1e-6, FAKE + 0x90000000,
                                       FAKE + 0xA0000000, FAKE + 0xB0000000, 1 << 30, None)

    def dec(st):
        return lib.gdn_decode_strided(ctypes.byref(B.make_shape(4, 8, 16, 32)), ctypes.byref(st), 2, 8, FAKE,
                                      FAKE + 0x10000000, FAKE + 0x20000000, FAKE + 0x30000000,
                                      FAKE + 0x40000000, FAKE + 0x50000000, FAKE + 0x60000000,
                                      FAKE + 0x70000000, None, None, None, 1e-6, FAKE + 0x90000000, None)
    for call in (pre, dec):
        assert call(strides(q=(16 * 128 + 4, 128))) == 1   # not a multiple of 8 elements
        assert call(strides(k=(16 * 128, 64))) == 1        # heads closer than a 128-element row
        assert call(strides(v=(0, 128))) == 1              # zero token stride
        assert call(strides(a=(32, 0))) == 1
    # a packed projection row: q | k | v | z | b | a, 12,352 elements per token
    W = 2 * 16 * 128 + 2 * 32 * 128 + 2 * 32
    packed = strides(q=(W, 128), k=(W, 128), v=(W, 128), z=(W, 128), a=(W, 1), b=(W, 1))
    # out must not lie inside the span of the packed inputs
    assert lib.gdn_prefill_strided(ctypes.byref(B.make_shape(1, 64, 16, 32)), ctypes.byref(packed), FAKE,
                                   FAKE + 4096, FAKE + 8192, FAKE + 24640, FAKE + 24576, FAKE + 0x50000000,
                                   FAKE + 0x60000000, None, FAKE + 0x80000000, None, None, 1e-6,
                                   FAKE + 64 * W, FAKE + 0xA0000000, FAKE + 0xB0000000, 1 << 30, None) == 1


def test_conv_entry_points_reject_bad_descriptors(lib):
    # host-side validation only: every call here fails before any launch
    W, S = FAKE + 0xC0000000, FAKE + 0xD0000000
    shape = B.make_shape(1, 64, 16, 32)

    def pre(width=4, weight=W, sin=S, sout=S, out=FAKE + 0x80000000):
        cv = B.Conv(width, weight, sin, sout)
        return lib.gdn_prefill_conv(ctypes.byref(shape), None, ctypes.byref(cv), FAKE, FAKE + 0x10000000,
                                    FAKE + 0x20000000, FAKE + 0x30000000, FAKE + 0x40000000, FAKE + 0x50000000,
                                    FAKE + 0x60000000, None, FAKE + 0x70000000, None, None, 1e-6, out,
                                    FAKE + 0x90000000, FAKE + 0xA0000000, 1 << 40, None)

    def dec(width=4, weight=W, sin=S, sout=S):
        cv = B.Conv(width, weight, sin, sout)
        return lib.gdn_decode_conv(ctypes.byref(B.make_shape(4, 8, 16, 32)), None, ctypes.byref(cv), 2, 8, FAKE,
                                   FAKE + 0x10000000, FAKE + 0x20000000, FAKE + 0x30000000, FAKE + 0x40000000,
                                   FAKE + 0x50000000, FAKE + 0x60000000, FAKE + 0x70000000, None, None, None,
                                   1e-6, FAKE + 0x90000000, None)
    for call in (pre, dec):
        assert call(width=0) == 1                    # width outside 1..4
        assert call(width=5) == 1
        assert call(weight=None) == 1
        assert call(weight=W + 8) == 3               # weights need 16-byte alignment
        assert call(sin=S + 8, sout=S + 8) == 3      # states need 16-byte alignment
        assert call(sout=S + 4096) == 1              # partial overlap of the two states
        assert call(sout=FAKE + 0x20000000) == 1     # written state over an input (v)
    assert pre(sout=FAKE + 0x80000000) == 1          # over the output
    assert pre(sout=FAKE + 0x90000000) == 1          # over the final states
    assert dec(sin=None, sout=None) == 1             # decode needs the slot pool of conv states
    assert dec(sout=FAKE + 0x70000000) == 1          # over the recurrent-state pool
    assert dec(sin=FAKE + 0x90000000, sout=FAKE + 0x90000000) == 1   # over the output
    # conv width 1 carries no state: NULL states are fine up to the launch,
    # which the fake pointers never reach in the other cases either
    assert pre(width=1, sin=None, sout=None, out=FAKE) == 1          # (out over q: still rejected)


def test_missing_library_fails_loudly(tmp_path):
    saved = B._lib
    try:
        B._lib = None
        with pytest.raises(ImportError):
            B.load(str(tmp_path / "nope.so"))
    finally:
        B._lib = saved


def _no_device():
    """True when no CUDA device is visible: then a call that passes every host
    check stops at the device lookup with GDN_ERR_CUDA, before any launch,
    which lets the tests below show that the one changed pointer is what a
    rejected call trips on.  (With a GPU present such a call would launch on
    the fake pointers, so it is never made.)"""
    import torch
    return not torch.cuda.is_available()


def test_prefill_rejects_writes_over_inputs(lib):
    """The workspace, out and final_state are written while the inputs are
    read: any overlap with an input is refused on the host (pegainfer page,
    Correctness: alias handling)."""
    ok = B.make_shape(1, 64, 16, 32)
    z, w = FAKE + 0xB0000000, FAKE + 0xC0000000
    if _no_device():
        assert _prefill(lib, ok) == 4                        # every host check passes
        assert _prefill(lib, ok, z=z, w=w) == 4
        assert _prefill(lib, ok, init=FAKE + 0x90000000) == 4   # in place: final_state == init_state
    for name, base in (("q", 0), ("k", 0x10000000), ("v", 0x20000000), ("a", 0x30000000), ("b", 0x40000000),
                       ("A_log", 0x50000000), ("dt_bias", 0x60000000), ("cu", 0x70000000)):
        assert _prefill(lib, ok, ws=FAKE + base) == 1, name            # workspace starts on the input
        assert _prefill(lib, ok, ws=FAKE + base - 0x400) == 1, name    # and one that ends in it
        assert _prefill(lib, ok, fin=FAKE + base) == 1, name           # final_state over the input
    assert _prefill(lib, ok, z=z, w=w, ws=z) == 1                      # workspace over z
    assert _prefill(lib, ok, z=z, w=w, ws=w - 0x400) == 1              # ... over the norm weights
    assert _prefill(lib, ok, z=z, w=w, fin=w) == 1                     # final_state over the norm weights
    assert _prefill(lib, ok, init=FAKE + 0xD0000000, ws=FAKE + 0xD0000000) == 1   # ... over init_state
    assert _prefill(lib, ok, init=FAKE + 0xD0000000, fin=FAKE + 0xD0000400) == 1  # partial state overlap
    assert _prefill(lib, ok, out=FAKE + 0xA0000000) == 1               # out over the workspace


def test_decode_rejects_a_pool_over_inputs(lib):
    def dec(shape, **kw):
        a = dict(q=FAKE, k=FAKE + 0x10000000, v=FAKE + 0x20000000, a=FAKE + 0x30000000,
                 b=FAKE + 0x40000000, A_log=FAKE + 0x50000000, dt=FAKE + 0x60000000,
                 state=FAKE + 0x70000000, idx=FAKE + 0x80000000, z=None, w=None, eps=1e-6,
                 out=FAKE + 0x90000000)
        a.update(kw)
        return lib.gdn_decode_slots(ctypes.byref(shape), 2, 8, a["q"], a["k"], a["v"], a["a"], a["b"], a["A_log"],
                                    a["dt"], a["state"], a["idx"], a["z"], a["w"], a["eps"], a["out"], None)
    sh = B.make_shape(4, 8, 16, 32)
    if _no_device():
        assert dec(sh) == 4
    for name, base in (("q", 0), ("v", 0x20000000), ("a", 0x30000000), ("A_log", 0x50000000),
                       ("dt_bias", 0x60000000), ("state_idx", 0x80000000)):
        assert dec(sh, state=FAKE + base) == 1, name
    assert dec(sh, z=FAKE + 0xA0000000, w=FAKE + 0xB0000000, state=FAKE + 0xA0000000) == 1   # over z


def test_prefill_conv_rejects_writes_over_its_weights(lib):
    W = FAKE + 0xC0000000
    shape = B.make_shape(1, 64, 16, 32)

    def pre(ws=FAKE + 0xA0000000, out=FAKE + 0x80000000, fin=FAKE + 0x90000000):
        cv = B.Conv(4, W, None, None)
        return lib.gdn_prefill_conv(ctypes.byref(shape), None, ctypes.byref(cv), FAKE, FAKE + 0x10000000,
                                    FAKE + 0x20000000, FAKE + 0x30000000, FAKE + 0x40000000, FAKE + 0x50000000,
                                    FAKE + 0x60000000, None, FAKE + 0x70000000, None, None, 1e-6, out, fin, ws,
                                    1 << 40, None)
    if _no_device():
        assert pre() == 4
    assert pre(ws=W) == 1
    assert pre(out=W) == 1
    assert pre(fin=W) == 1


def test_conv_prefill_rejects_bad_arguments(lib):
    """gdn_conv_prefill writes y only: a state_out, a y over an input, or a
    bad descriptor is refused on the host."""
    W, S = FAKE + 0xC0000000, FAKE + 0xD0000000
    shape = B.make_shape(1, 64, 16, 32)

    def call(width=4, weight=W, sin=S, sout=None, y=FAKE + 0x80000000, cu=FAKE + 0x70000000):
        cv = B.Conv(width, weight, sin, sout)
        return lib.gdn_conv_prefill(ctypes.byref(shape), None, ctypes.byref(cv), FAKE, FAKE + 0x10000000,
                                    FAKE + 0x20000000, cu, y, None)
    if _no_device():
        assert call() == 4                    # every host check passes
    assert call(sout=S) == 1                  # this entry point writes no state
    assert call(width=0) == 1
    assert call(weight=None) == 1
    assert call(cu=None) == 1
    assert call(y=None) == 1
    assert call(y=FAKE + 0x20000000) == 1     # y over v
    assert call(y=W) == 1                     # y over the weights
    assert call(y=FAKE + 0x80000000 + 8) == 3
