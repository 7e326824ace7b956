"""fp64 CPU oracle for the Gated DeltaNet layer core (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may use this package; the product path
(``gated_deltanet_linear_08_gb300``) never imports it and shares no code with
it.  See ``gdn_oracle.c`` for what each function computes and which passage of
the pages it follows.

Parity status of each function (what pins it, see tests/test_oracle.py):
  prep                 softplus/sigmoid/L2 norm against ``math`` on a grid.
  core                 closed forms (T=1, pure decay, exact replacement), a
                       dense transition-matrix brute force, split-sequence
                       carry, varlen packing.
  core_chunked         equal to ``core`` at chunk boundaries 1..200.
  gated_rmsnorm        unit RMS after dividing out w*silu(z); hand-computed
                       fixture.
  prefill / decode     compositions of the above.
The grouped-head mapping (v head h reads k head h // (Hv/Hk)), the L2-norm
epsilon 1e-6 and the per-head gated-norm grouping are readings of the pages,
not facts they print: parity of those choices is unpinned by the pages.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None
L2_EPS = 1e-6


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
            "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.gdn_oracle_softplus.argtypes = [f64]
            lib.gdn_oracle_softplus.restype = f64
            lib.gdn_oracle_sigmoid.argtypes = [f64]
            lib.gdn_oracle_sigmoid.restype = f64
            lib.gdn_oracle_prep.argtypes = [i64, i32, i32, i32, P, P, P, P, P, P, f64,
                                            P, P, P, P]
            lib.gdn_oracle_prep.restype = None
            lib.gdn_oracle_gated_rmsnorm.argtypes = [i64, i32, P, P, P, f64]
            lib.gdn_oracle_gated_rmsnorm.restype = None
            lib.gdn_oracle_core.argtypes = [i32, P, i32, i32, i32, i32, P, P, P, P, P, P,
                                            P, P, i32]
            lib.gdn_oracle_core.restype = i32
            lib.gdn_oracle_core_chunked.argtypes = [i32, P, i32, i32, i32, i32, i32, P, P,
                                                    P, P, P, P, P, P, i32]
            lib.gdn_oracle_core_chunked.restype = i32
            lib.gdn_oracle_prefill.argtypes = [i32, P, i32, i32, i32, i32, P, P, P, P, P,
                                               P, P, f64, P, P, P, f64, P, P, i32]
            lib.gdn_oracle_prefill.restype = i32
            lib.gdn_oracle_decode_step.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P,
                                                   P, P, f64, P, P, P, f64, P, i32]
            lib.gdn_oracle_decode_step.restype = i32
            _lib = lib
    return _lib


def _c(x, dtype=np.float64):
    """Contiguous array of the given dtype (None passes through)."""
    if x is None:
        return None
    return np.ascontiguousarray(x, dtype=dtype)


def _p(x):
    return None if x is None else x.ctypes.data_as(ctypes.c_void_p)


def softplus(x: float) -> float:
    return _load().gdn_oracle_softplus(float(x))


def sigmoid(x: float) -> float:
    return _load().gdn_oracle_sigmoid(float(x))


def prep(q, k, a, b, A_log, dt_bias, l2_eps: float = L2_EPS):
    """Gate g, beta, and L2-normalised q/k.  Shapes: q,k [T,hk,dk]; a,b [T,hv]."""
    q, k, a, b = _c(q), _c(k), _c(a), _c(b)
    A_log, dt_bias = _c(A_log), _c(dt_bias)
    T, hk, dk = q.shape
    hv = a.shape[1]
    g = np.empty((T, hv)); beta = np.empty((T, hv))
    qn = np.empty_like(q); kn = np.empty_like(k)
    _load().gdn_oracle_prep(T, hk, hv, dk, _p(q), _p(k), _p(a), _p(b), _p(A_log),
                            _p(dt_bias), float(l2_eps), _p(g), _p(beta), _p(qn), _p(kn))
    return g, beta, qn, kn


def gated_rmsnorm(o, z, w, eps: float):
    """y = o / sqrt(mean(o^2) + eps) * w * silu(z) over the last axis."""
    o = np.array(o, dtype=np.float64, order="C", copy=True)
    z, w = _c(z), _c(w)
    dv = o.shape[-1]
    _load().gdn_oracle_gated_rmsnorm(o.size // dv, dv, _p(o), _p(z), _p(w), float(eps))
    return o


def core(cu_seqlens, g, beta, qn, kn, v, init_state=None, nthreads: int = 0):
    """Token-by-token recurrence on prepped inputs; returns (out, final_state)."""
    cu = _c(cu_seqlens, np.int32)
    g, beta, qn, kn, v = _c(g), _c(beta), _c(qn), _c(kn), _c(v)
    init_state = _c(init_state)
    N = cu.shape[0] - 1
    T, hk, dk = qn.shape
    hv, dv = v.shape[1], v.shape[2]
    out = np.zeros((T, hv, dv))
    fin = np.zeros((N, hv, dk, dv))
    rc = _load().gdn_oracle_core(N, _p(cu), hk, hv, dk, dv, _p(g), _p(beta), _p(qn), _p(kn),
                                 _p(v), _p(init_state), _p(out), _p(fin), int(nthreads))
    if rc != 0:
        raise ValueError("oracle core: bad arguments")
    return out, fin


def core_chunked(cu_seqlens, g, beta, qn, kn, v, init_state=None, chunk: int = 64,
                 nthreads: int = 0):
    """Chunked (WY/UT) fp64 form of ``core``; returns (out, final_state)."""
    cu = _c(cu_seqlens, np.int32)
    g, beta, qn, kn, v = _c(g), _c(beta), _c(qn), _c(kn), _c(v)
    init_state = _c(init_state)
    N = cu.shape[0] - 1
    T, hk, dk = qn.shape
    hv, dv = v.shape[1], v.shape[2]
    out = np.zeros((T, hv, dv))
    fin = np.zeros((N, hv, dk, dv))
    rc = _load().gdn_oracle_core_chunked(N, _p(cu), hk, hv, dk, dv, int(chunk), _p(g),
                                         _p(beta), _p(qn), _p(kn), _p(v), _p(init_state),
                                         _p(out), _p(fin), int(nthreads))
    if rc != 0:
        raise ValueError("oracle core_chunked: bad arguments")
    return out, fin


def prefill(cu_seqlens, q, k, v, a, b, A_log, dt_bias, init_state=None, z=None,
            norm_w=None, eps: float = 1e-6, l2_eps: float = L2_EPS, nthreads: int = 0):
    """Full prefill on raw (bf16-valued) inputs; returns (out, final_state)."""
    cu = _c(cu_seqlens, np.int32)
    q, k, v, a, b = _c(q), _c(k), _c(v), _c(a), _c(b)
    A_log, dt_bias = _c(A_log), _c(dt_bias)
    init_state, z, norm_w = _c(init_state), _c(z), _c(norm_w)
    if z is not None and norm_w is None:
        raise ValueError("oracle prefill: z given without norm_w")
    N = cu.shape[0] - 1
    T, hk, dk = q.shape
    hv, dv = v.shape[1], v.shape[2]
    out = np.zeros((T, hv, dv))
    fin = np.zeros((N, hv, dk, dv))
    rc = _load().gdn_oracle_prefill(N, _p(cu), hk, hv, dk, dv, _p(q), _p(k), _p(v), _p(a),
                                    _p(b), _p(A_log), _p(dt_bias), float(l2_eps),
                                    _p(init_state), _p(z), _p(norm_w), float(eps), _p(out),
                                    _p(fin), int(nthreads))
    if rc != 0:
        raise ValueError("oracle prefill: bad arguments")
    return out, fin


def decode_step(q, k, v, a, b, A_log, dt_bias, state, z=None, norm_w=None,
                eps: float = 1e-6, l2_eps: float = L2_EPS, nthreads: int = 0):
    """One decode token per sequence.  ``state`` (float64, C-contiguous) is
    updated in place; returns out [B, hv, dv]."""
    if not (isinstance(state, np.ndarray) and state.dtype == np.float64
            and state.flags["C_CONTIGUOUS"]):
        raise TypeError("oracle decode_step: state must be a C-contiguous float64 array")
    q, k, v, a, b = _c(q), _c(k), _c(v), _c(a), _c(b)
    A_log, dt_bias, z, norm_w = _c(A_log), _c(dt_bias), _c(z), _c(norm_w)
    B, hk, dk = q.shape
    hv, dv = v.shape[1], v.shape[2]
    out = np.zeros((B, hv, dv))
    rc = _load().gdn_oracle_decode_step(B, hk, hv, dk, dv, _p(q), _p(k), _p(v), _p(a),
                                        _p(b), _p(A_log), _p(dt_bias), float(l2_eps),
                                        _p(state), _p(z), _p(norm_w), float(eps), _p(out),
                                        int(nthreads))
    if rc != 0:
        raise ValueError("oracle decode_step: bad arguments")
    return out
