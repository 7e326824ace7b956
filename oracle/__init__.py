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
  causal_conv_silu /   impulse weights reduce it to shifted inputs, numpy's
  conv_inputs          np.convolve per channel, split-sequence state carry;
                       the conv itself is a reading (nothing on the pages
                       defines it), so its parity is unpinned by the pages.
The grouped-head mapping (v head h reads k head h // (Hv/Hk)), the L2-norm
epsilon 1e-6 and the per-head gated-norm grouping are readings of the pages,
not facts they print: parity of those choices is unpinned by the pages.
"""
from __future__ import annotations

import contextlib
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


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle with gcc (OpenMP when available, no fast-math).
    ``src``/``out`` build another copy of the source: the mutation test
    compiles the oracle with one planted mistake that way."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
            "-shared", "-fPIC", "-o", tmp, src, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, out)
    return out


def _configure(lib):
    """Declare the C signatures on a loaded oracle library."""
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
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _configure(ctypes.CDLL(_LIB_PATH))
    return _lib


@contextlib.contextmanager
def library(path: str):
    """Inside the block every function of this module runs on the library at
    ``path`` (another build of the oracle's source, e.g. a planted mistake)."""
    global _lib
    lib = _configure(ctypes.CDLL(path))
    with _lock:
        old, _lib = _lib, lib
    try:
        yield
    finally:
        with _lock:
            _lib = old


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


# ---------------------------------------------------------------------------
# Causal conv1d + SiLU ahead of the core.  The JevAny page ("Add opt-in fused
# Qwen3.5 inference kernels", Measurements) lists causal-conv1d among the
# path's dependencies but does not define it; the definition below is a
# reading (plain numpy, fp64):
#   * channels: q | k | v of a token, Hk*128 + Hk*128 + Hv*128 of them;
#   * per channel c a causal window of width K (1..4) with weights w[c, 0..K-1]:
#         y[t, c] = silu( sum_j w[c, j] * x[t - (K-1) + j, c] )
#     where positions before the sequence start come from the carried state
#     (the K-1 raw inputs that preceded it, oldest first) or are zero;
#   * y is rounded to bf16 (round to nearest even), as a separate conv pass
#     would write it, and the core then runs on those values;
#   * the new state is the sequence's last K-1 raw inputs (state rows first
#     when the sequence is shorter than K-1).
# ---------------------------------------------------------------------------
def round_bf16(x):
    """Round fp64 values to the nearest bf16 value (ties to even); finite
    inputs in the normal range, as on the path."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                    # x = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)   # 8 significant bits


def silu(x):
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def causal_conv_silu(x, w, state=None):
    """One sequence: x [T, C] raw inputs, w [C, K], state [K-1, C] or None.
    Returns (y [T, C] bf16-rounded, new state [K-1, C])."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    T, C = x.shape
    K = w.shape[1]
    prev = np.zeros((K - 1, C)) if state is None else np.asarray(state, dtype=np.float64)
    xe = np.concatenate([prev, x], axis=0)          # [K-1+T, C]
    acc = np.zeros((T, C))
    for j in range(K):
        acc += w[:, j][None, :] * xe[j:j + T]
    return round_bf16(silu(acc)), xe[T:T + K - 1] if K > 1 else np.zeros((0, C))


def conv_inputs(cu_seqlens, q, k, v, w, state=None):
    """The conv over packed sequences: q, k [T, Hk, D], v [T, Hv, D], w
    [Hk*D + Hk*D + Hv*D, K], state [N, K-1, C] or None.  Returns the post-conv
    q, k, v (bf16-rounded fp64) and the new states [N, K-1, C]."""
    cu = np.asarray(cu_seqlens)
    T, hk, d = q.shape
    hv = v.shape[1]
    x = np.concatenate([np.asarray(q, np.float64).reshape(T, -1), np.asarray(k, np.float64).reshape(T, -1),
                        np.asarray(v, np.float64).reshape(T, -1)], axis=1)
    C, K = x.shape[1], np.asarray(w).shape[1]
    y = np.zeros_like(x)
    new = np.zeros((len(cu) - 1, K - 1, C))
    for n in range(len(cu) - 1):
        s, e = cu[n], cu[n + 1]
        y[s:e], new[n] = causal_conv_silu(x[s:e], w, None if state is None else state[n])
    qc = y[:, :hk * d].reshape(T, hk, d)
    kc = y[:, hk * d:2 * hk * d].reshape(T, hk, d)
    vc = y[:, 2 * hk * d:].reshape(T, hv, d)
    return qc, kc, vc, new
