"""ctypes binding of libgdn (include/gdn.h): argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this module
checks dtypes/devices/shapes of torch tensors, passes raw device pointers and
the current CUDA stream, and turns status codes into exceptions.  It never
falls back to another implementation: if the library is missing, loading
raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libgdn.so")
_lock = threading.Lock()
_lib = None

GDN_OK = 0
STATUS_NAMES = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_UNSUPPORTED",
                3: "GDN_ERR_ALIGNMENT", 4: "GDN_ERR_CUDA", 5: "GDN_ERR_DEVICE_STATUS",
                6: "GDN_ERR_WORKSPACE"}
EXPORTED = ("gdn_status_string", "gdn_prefill_workspace_bytes", "gdn_prefill", "gdn_decode",
            "gdn_check_device_status", "gdn_prefill_noalloc", "gdn_decode_slots", "gdn_prefill_strided",
            "gdn_decode_strided", "gdn_prefill_conv", "gdn_decode_conv", "gdn_prefill_conv_workspace_bytes",
            "gdn_conv_prefill")


class GdnError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(msg)
        self.code = code


class Shape(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("total_tokens", ctypes.c_int32),
                ("hq", ctypes.c_int32), ("hk", ctypes.c_int32), ("hv", ctypes.c_int32),
                ("dk", ctypes.c_int32), ("dv", ctypes.c_int32)]


class Stride(ctypes.Structure):
    _fields_ = [("token", ctypes.c_int64), ("head", ctypes.c_int64)]


class Strides(ctypes.Structure):
    _fields_ = [("q", Stride), ("k", Stride), ("v", Stride), ("z", Stride), ("a", Stride), ("b", Stride)]


class Conv(ctypes.Structure):
    _fields_ = [("width", ctypes.c_int32), ("weight", ctypes.c_void_p), ("state_in", ctypes.c_void_p),
                ("state_out", ctypes.c_void_p)]


def load(path: Optional[str] = None):
    """Load libgdn.so (built by ``build.build()``); raises if it is absent."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise ImportError(
                    f"libgdn.so not found at {p}: build it with "
                    "gated_deltanet_linear_08_gb300.build.build() (needs nvcc)")
            lib = ctypes.CDLL(p)
            P, f32, sz = ctypes.c_void_p, ctypes.c_float, ctypes.c_size_t
            lib.gdn_status_string.argtypes = [ctypes.c_int]
            lib.gdn_status_string.restype = ctypes.c_char_p
            lib.gdn_prefill_workspace_bytes.argtypes = [ctypes.POINTER(Shape)]
            lib.gdn_prefill_workspace_bytes.restype = sz
            lib.gdn_prefill.argtypes = [ctypes.POINTER(Shape), P, P, P, P, P, P, P, P, P, P, P,
                                        f32, P, P, P, sz, P]
            lib.gdn_prefill.restype = ctypes.c_int
            lib.gdn_decode.argtypes = [ctypes.POINTER(Shape), P, P, P, P, P, P, P, P, P, P, f32,
                                       P, P]
            lib.gdn_decode.restype = ctypes.c_int
            lib.gdn_prefill_noalloc.argtypes = [ctypes.POINTER(Shape), P, P, P, P, P, P, P, P, P,
                                                P, P, f32, P, P, P]
            lib.gdn_prefill_noalloc.restype = ctypes.c_int
            lib.gdn_decode_slots.argtypes = [ctypes.POINTER(Shape), ctypes.c_int32, ctypes.c_int32, P, P, P, P,
                                             P, P, P, P, P, P, P, f32, P, P]
            lib.gdn_decode_slots.restype = ctypes.c_int
            lib.gdn_prefill_strided.argtypes = [ctypes.POINTER(Shape), ctypes.POINTER(Strides), P, P, P, P, P, P,
                                                P, P, P, P, P, f32, P, P, P, sz, P]
            lib.gdn_prefill_strided.restype = ctypes.c_int
            lib.gdn_decode_strided.argtypes = [ctypes.POINTER(Shape), ctypes.POINTER(Strides), ctypes.c_int32,
                                               ctypes.c_int32, P, P, P, P, P, P, P, P, P, P, P, f32, P, P]
            lib.gdn_decode_strided.restype = ctypes.c_int
            lib.gdn_prefill_conv_workspace_bytes.argtypes = [ctypes.POINTER(Shape)]
            lib.gdn_prefill_conv_workspace_bytes.restype = sz
            lib.gdn_prefill_conv.argtypes = [ctypes.POINTER(Shape), ctypes.POINTER(Strides), ctypes.POINTER(Conv),
                                             P, P, P, P, P, P, P, P, P, P, P, f32, P, P, P, sz, P]
            lib.gdn_prefill_conv.restype = ctypes.c_int
            lib.gdn_decode_conv.argtypes = [ctypes.POINTER(Shape), ctypes.POINTER(Strides), ctypes.POINTER(Conv),
                                            ctypes.c_int32, ctypes.c_int32, P, P, P, P, P, P, P, P, P, P, P, f32,
                                            P, P]
            lib.gdn_decode_conv.restype = ctypes.c_int
            lib.gdn_conv_prefill.argtypes = [ctypes.POINTER(Shape), ctypes.POINTER(Strides), ctypes.POINTER(Conv),
                                             P, P, P, P, P, P]
            lib.gdn_conv_prefill.restype = ctypes.c_int
            lib.gdn_check_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
            lib.gdn_check_device_status.restype = ctypes.c_int
            _lib = lib
    return _lib


def status_string(code: int) -> str:
    return load().gdn_status_string(int(code)).decode()


def _check(code: int):
    if code != GDN_OK:
        raise GdnError(code, status_string(code))


def make_shape(num_seqs: int, total_tokens: int, hk: int, hv: int, hq: Optional[int] = None,
               dk: int = 128, dv: int = 128) -> Shape:
    return Shape(num_seqs, total_tokens, hk if hq is None else hq, hk, hv, dk, dv)


def workspace_bytes(num_seqs: int, total_tokens: int, hk: int, hv: int, conv: bool = False) -> int:
    """Workspace of gdn_prefill, or with ``conv`` of gdn_prefill_conv."""
    s = make_shape(num_seqs, total_tokens, hk, hv)
    if conv:
        return int(load().gdn_prefill_conv_workspace_bytes(ctypes.byref(s)))
    return int(load().gdn_prefill_workspace_bytes(ctypes.byref(s)))


def _ptr(t: Optional[torch.Tensor], dtype, name: str, device) -> Optional[int]:
    if t is None:
        return None
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name}: expected device {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return t.data_ptr()


def _in_ptr(t: Optional[torch.Tensor], name: str, device) -> Optional[int]:
    """Pointer of a token input that may be a strided view (innermost
    dimension contiguous): checked by the library against its strides."""
    if t is None:
        return None
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name}: expected torch.bfloat16, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name}: expected device {device}, got {t.device}")
    if t.stride(-1) != 1:
        raise ValueError(f"{name}: the innermost dimension must be contiguous")
    return t.data_ptr()


def _token_strides(t: Optional[torch.Tensor], lead: int, name: str):
    """(token, head) element strides of a [tokens..., heads(, 128)] view whose
    `lead` leading dimensions flatten into the token index."""
    if t is None:
        return (0, 0)
    st, sh = t.stride(lead - 1), t.stride(lead)
    for d in range(lead - 1):   # the leading dimensions must flatten evenly
        if t.stride(d) != t.stride(d + 1) * t.shape[d + 1]:
            raise ValueError(f"{name}: the token dimensions do not flatten into one stride")
    return (st, sh)


def _strides(tensors: dict, lead: int):
    """None when every token input is dense, else the Strides structure."""
    if all(t is None or t.is_contiguous() for t in tensors.values()):
        return None
    s = Strides()
    for n in ("q", "k", "v", "z", "a", "b"):
        tok, head = _token_strides(tensors.get(n), lead, n)
        setattr(s, n, Stride(tok, head))
    return s


def _stream_handle(stream: Optional[torch.cuda.Stream], device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def alloc_workspace(num_seqs: int, total_tokens: int, hk: int, hv: int, device, conv: bool = False) -> torch.Tensor:
    """Device workspace for gdn_prefill (with ``conv``: gdn_prefill_conv);
    a torch allocation, 1024-byte aligned."""
    n = workspace_bytes(num_seqs, total_tokens, hk, hv, conv)
    buf = torch.empty(n + 1024, dtype=torch.uint8, device=device)
    off = (-buf.data_ptr()) % 1024
    return buf[off:off + n] if n else buf[:0]


def _conv(weight, state_in, state_out, dev):
    """The conv descriptor of gdn_conv_t (weight [C, K] bf16, states [rows, K-1, C] bf16)."""
    if weight.dim() != 2:
        raise ValueError("conv_weight must be [channels, width]")
    bf = torch.bfloat16
    return Conv(int(weight.shape[1]), _ptr(weight, bf, "conv_weight", dev), _ptr(state_in, bf, "conv_state", dev),
                _ptr(state_out, bf, "conv_state_out", dev))


def prefill(q, k, v, a, b, A_log, dt_bias, cu_seqlens, init_state=None, z=None, norm_w=None,
            eps: float = 1e-6, out=None, final_state=None, workspace=None, stream=None,
            conv_weight=None, conv_state=None, conv_state_out=None):
    """Chunked GDN prefill through ``gdn_prefill``.  Returns (out, final_state),
    or (out, final_state, conv_state_out) when ``conv_weight`` is given.

    With ``conv_weight`` [Hk*128 + Hk*128 + Hv*128, K] bf16 the causal conv1d
    + SiLU runs on q | k | v ahead of the core (``gdn_prefill_conv``), from
    ``conv_state`` [N, K-1, C] bf16 (None: zeros); ``conv_state_out`` (may be
    ``conv_state`` itself) receives each sequence's last K-1 raw inputs.

    q, k [T, Hk, 128] bf16; v [T, Hv, 128] bf16; a, b [T, Hv] bf16 (dense,
    or views with a contiguous innermost dimension, e.g. slices of one packed
    projection output, passed as strides); A_log, dt_bias [Hv] fp32; cu_seqlens [N+1] int32 (device); init_state
    [N, Hv, 128, 128] fp32 or None; z [T, Hv, 128] bf16 and norm_w [128] bf16
    for the gated-RMSNorm epilogue.  ``final_state`` may be ``init_state``.
    """
    dev = q.device
    T, hk = q.shape[0], q.shape[1]
    hv = v.shape[1]
    N = cu_seqlens.shape[0] - 1
    if out is None:
        out = torch.empty(T, hv, 128, dtype=torch.bfloat16, device=dev)
    if final_state is None:
        final_state = torch.empty(N, hv, 128, 128, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(N, T, hk, hv, dev, conv=conv_weight is not None)
    bf, f32 = torch.bfloat16, torch.float32
    shape = make_shape(N, T, hk, hv)
    strides = _strides(dict(q=q, k=k, v=v, z=z, a=a, b=b), 1)
    ins = [_in_ptr(t, n, dev) for t, n in ((q, "q"), (k, "k"), (v, "v"), (a, "a"), (b, "b"))]
    rest = (_ptr(A_log, f32, "A_log", dev), _ptr(dt_bias, f32, "dt_bias", dev),
            _ptr(init_state, f32, "init_state", dev), _ptr(cu_seqlens, torch.int32, "cu_seqlens", dev),
            _in_ptr(z, "z", dev), _ptr(norm_w, bf, "norm_w", dev), float(eps), _ptr(out, bf, "out", dev),
            _ptr(final_state, f32, "final_state", dev), _ptr(workspace, torch.uint8, "workspace", dev),
            int(workspace.numel()), _stream_handle(stream, dev))
    if conv_weight is not None:
        K = int(conv_weight.shape[1])
        if conv_state_out is None:
            conv_state_out = torch.empty(N, K - 1, conv_weight.shape[0], dtype=torch.bfloat16, device=dev)
        conv = _conv(conv_weight, conv_state, conv_state_out, dev)
        code = load().gdn_prefill_conv(ctypes.byref(shape), None if strides is None else ctypes.byref(strides),
                                       ctypes.byref(conv), *ins, *rest)
        _check(code)
        return out, final_state, conv_state_out
    if strides is None:
        code = load().gdn_prefill(ctypes.byref(shape), *ins, *rest)
    else:
        code = load().gdn_prefill_strided(ctypes.byref(shape), ctypes.byref(strides), *ins, *rest)
    _check(code)
    return out, final_state


def conv_prefill(q, k, v, cu_seqlens, conv_weight, conv_state=None, y=None, stream=None):
    """The causal conv1d + SiLU alone through ``gdn_conv_prefill``: returns y
    [T, Hk*128 + Hk*128 + Hv*128] bf16, the q | k | v rows the prefill's conv
    feeds to the core (bit for bit).  q, k [T, Hk, 128], v [T, Hv, 128] bf16;
    conv_weight [C, K] bf16; conv_state [N, K-1, C] bf16 or None (zeros)."""
    dev = q.device
    T, hk = q.shape[0], q.shape[1]
    hv = v.shape[1]
    N = cu_seqlens.shape[0] - 1
    C = conv_weight.shape[0]
    if y is None:
        y = torch.empty(T, C, dtype=torch.bfloat16, device=dev)
    shape = make_shape(N, T, hk, hv)
    strides = _strides(dict(q=q, k=k, v=v, z=None, a=None, b=None), 1)
    conv = _conv(conv_weight, conv_state, None, dev)
    code = load().gdn_conv_prefill(ctypes.byref(shape), None if strides is None else ctypes.byref(strides),
                                   ctypes.byref(conv), _in_ptr(q, "q", dev), _in_ptr(k, "k", dev),
                                   _in_ptr(v, "v", dev), _ptr(cu_seqlens, torch.int32, "cu_seqlens", dev),
                                   _ptr(y, torch.bfloat16, "y", dev), _stream_handle(stream, dev))
    _check(code)
    return y


def prefill_noalloc(q, k, v, a, b, A_log, dt_bias, cu_seqlens, init_state=None, z=None,
                    norm_w=None, eps: float = 1e-6, out=None, final_state=None, stream=None):
    """Prefill through ``gdn_prefill_noalloc``: the library's own fixed scratch
    instead of a workspace, for callers that cannot allocate device memory.
    ``out`` and ``final_state`` should be passed in by such callers (the
    defaults here allocate them with torch for convenience)."""
    dev = q.device
    T, hk = q.shape[0], q.shape[1]
    hv = v.shape[1]
    N = cu_seqlens.shape[0] - 1
    if out is None:
        out = torch.empty(T, hv, 128, dtype=torch.bfloat16, device=dev)
    if final_state is None:
        final_state = torch.empty(N, hv, 128, 128, dtype=torch.float32, device=dev)
    bf, f32 = torch.bfloat16, torch.float32
    shape = make_shape(N, T, hk, hv)
    code = load().gdn_prefill_noalloc(
        ctypes.byref(shape), _ptr(q, bf, "q", dev), _ptr(k, bf, "k", dev), _ptr(v, bf, "v", dev),
        _ptr(a, bf, "a", dev), _ptr(b, bf, "b", dev), _ptr(A_log, f32, "A_log", dev),
        _ptr(dt_bias, f32, "dt_bias", dev), _ptr(init_state, f32, "init_state", dev),
        _ptr(cu_seqlens, torch.int32, "cu_seqlens", dev), _ptr(z, bf, "z", dev),
        _ptr(norm_w, bf, "norm_w", dev), float(eps), _ptr(out, bf, "out", dev),
        _ptr(final_state, f32, "final_state", dev), _stream_handle(stream, dev))
    _check(code)
    return out, final_state


def decode(q, k, v, a, b, A_log, dt_bias, state, z=None, norm_w=None, eps: float = 1e-6,
           out=None, stream=None):
    """One decode token per sequence through ``gdn_decode``; ``state`` is
    updated in place.  Returns out [B, Hv, 128] bf16."""
    dev = q.device
    B, hk = q.shape[0], q.shape[1]
    hv = v.shape[1]
    if out is None:
        out = torch.empty(B, hv, 128, dtype=torch.bfloat16, device=dev)
    bf, f32 = torch.bfloat16, torch.float32
    shape = make_shape(B, B, hk, hv)
    code = load().gdn_decode(
        ctypes.byref(shape), _ptr(q, bf, "q", dev), _ptr(k, bf, "k", dev), _ptr(v, bf, "v", dev),
        _ptr(a, bf, "a", dev), _ptr(b, bf, "b", dev), _ptr(A_log, f32, "A_log", dev),
        _ptr(dt_bias, f32, "dt_bias", dev), _ptr(state, f32, "state", dev),
        _ptr(z, bf, "z", dev), _ptr(norm_w, bf, "norm_w", dev), float(eps),
        _ptr(out, bf, "out", dev), _stream_handle(stream, dev))
    _check(code)
    return out


def decode_slots(q, k, v, a, b, A_log, dt_bias, state_pool, state_idx=None, z=None, norm_w=None,
                 eps: float = 1e-6, out=None, stream=None, conv_weight=None, conv_state=None,
                 conv_state_out=None):
    """``tokens`` consecutive tokens per sequence through ``gdn_decode_slots``;
    the pool slots named by ``state_idx`` are updated in place.  With
    ``conv_weight`` [C, K] bf16 the causal conv1d + SiLU runs ahead of the
    core (``gdn_decode_conv``) and ``conv_state`` [P, K-1, C] bf16, a pool
    indexed like ``state_pool``, is rolled in place -- or, given
    ``conv_state_out`` (a second pool), written there by the decode kernel.

    q, k [B, T, Hk, 128] bf16; v [B, T, Hv, 128] bf16; a, b [B, T, Hv] bf16;
    state_pool [P, Hv, 128, 128] fp32; state_idx [B] int32 (device) or None
    for slot n; z [B, T, Hv, 128] bf16 and norm_w [128] bf16 for the gated
    RMSNorm.  Returns out [B, T, Hv, 128] bf16.
    """
    dev = q.device
    B, T, hk = q.shape[0], q.shape[1], q.shape[2]
    hv = v.shape[2]
    if out is None:
        out = torch.empty(B, T, hv, 128, dtype=torch.bfloat16, device=dev)
    bf, f32 = torch.bfloat16, torch.float32
    shape = make_shape(B, B * T, hk, hv)
    strides = _strides(dict(q=q, k=k, v=v, z=z, a=a, b=b), 2)
    ins = [_in_ptr(t, n, dev) for t, n in ((q, "q"), (k, "k"), (v, "v"), (a, "a"), (b, "b"))]
    rest = (_ptr(A_log, f32, "A_log", dev), _ptr(dt_bias, f32, "dt_bias", dev),
            _ptr(state_pool, f32, "state_pool", dev), _ptr(state_idx, torch.int32, "state_idx", dev),
            _in_ptr(z, "z", dev), _ptr(norm_w, bf, "norm_w", dev), float(eps), _ptr(out, bf, "out", dev),
            _stream_handle(stream, dev))
    if conv_weight is not None:
        conv = _conv(conv_weight, conv_state, conv_state if conv_state_out is None else conv_state_out, dev)
        code = load().gdn_decode_conv(ctypes.byref(shape), None if strides is None else ctypes.byref(strides),
                                      ctypes.byref(conv), int(T), int(state_pool.shape[0]), *ins, *rest)
    elif strides is None:
        code = load().gdn_decode_slots(ctypes.byref(shape), int(T), int(state_pool.shape[0]), *ins, *rest)
    else:
        code = load().gdn_decode_strided(ctypes.byref(shape), ctypes.byref(strides), int(T),
                                         int(state_pool.shape[0]), *ins, *rest)
    _check(code)
    return out


def check_device_status() -> int:
    """Synchronise and read/clear the kernels' status bits (0 = clean)."""
    bits = ctypes.c_uint32(0)
    code = load().gdn_check_device_status(ctypes.byref(bits))
    if code not in (GDN_OK, 5):
        _check(code)
    return int(bits.value)
