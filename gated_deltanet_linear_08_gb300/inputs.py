"""Seeded synthetic inputs for the Gated DeltaNet layer core.

This module only draws random numbers; it holds none of the method's
arithmetic.  Both the fp64 oracle (under ``oracle/``) and the CUDA path are fed
from here, so the two sides see identical bits.

Shapes and distributions follow the Qwen3.5-4B geometry named on the pegainfer
page ("feat(qwen35): add SM120 FlashInfer GDN prefill candidate", section
Correctness: Hq/Hk/Hv/D = 16/16/32/128) and the grouped-value Hv=48 member of
the same family ("Hv48 generalization", same section).

Draw order (one ``torch.Generator`` seeded once per case):
  1. varlen sequence lengths (only for cases that draw them);
  2. q, k, v, a, b ~ N(0, 1) in fp32, then rounded to bf16;
  3. A_log = log(U(1, 16)) in fp32;
  4. dt_bias ~ N(0, 1) in fp32;
  5. initial states ~ N(0, 0.1) (standard deviation 0.1) in fp32, if any;
  6. z ~ N(0, 1) rounded to bf16 and w ~ N(1, 0.1) rounded to bf16, if the
     gated-RMSNorm epilogue is on.
Decode cases draw A_log, dt_bias and the states first, then q, k, v, a, b step
by step from the same stream.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import torch

D_HEAD = 128
CHUNK = 64


@dataclass
class PrefillCase:
    """One prefill workload: packed sequences over a grouped-head geometry."""

    name: str
    seqlens: Optional[List[int]] = None  # None -> drawn (see n_random_seqs)
    n_random_seqs: int = 0               # draw this many lengths in [1, max_random_len]
    max_random_len: int = 1024
    hk: int = 16
    hv: int = 32
    d: int = D_HEAD
    init_state: bool = False
    gated_norm: bool = False
    eps: float = 1e-6
    seed: int = 0
    # Overrides for extra parity cases (weak decay, pure decay, ...).
    a_log_const: Optional[float] = None  # A_log filled with this value
    b_const: Optional[float] = None      # b filled with this value (before bf16)


@dataclass
class DecodeCase:
    """Decode workload: ``batch`` independent sequences, one token per step."""

    name: str
    batch: int = 256
    hk: int = 16
    hv: int = 32
    d: int = D_HEAD
    steps: int = 64
    gated_norm: bool = False
    eps: float = 1e-6
    seed: int = 0


@dataclass
class DecodeSlotsCase:
    """Decode of ``tokens`` consecutive tokens per sequence against a pool of
    ``slots`` recurrent states.  Sequence n uses a distinct random slot;
    ``skipped`` of them carry slot -1 and ``out_of_pool`` carry slot ``slots``
    (past the pool)."""

    name: str
    batch: int = 64
    tokens: int = 4
    slots: int = 96
    skipped: int = 0
    out_of_pool: int = 0
    hk: int = 16
    hv: int = 32
    d: int = D_HEAD
    gated_norm: bool = False
    eps: float = 1e-6
    seed: int = 0


def _bf16(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16)


def make_prefill_inputs(case: PrefillCase) -> dict:
    """Return CPU tensors for one prefill case (see module docstring for order)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(case.seed)
    if case.seqlens is None:
        lens = torch.randint(1, case.max_random_len + 1, (case.n_random_seqs,), generator=g)
        seqlens = [int(x) for x in lens]
    else:
        seqlens = list(case.seqlens)
    n = len(seqlens)
    t_tot = sum(seqlens)
    cu = torch.zeros(n + 1, dtype=torch.int32)
    if n:
        cu[1:] = torch.cumsum(torch.tensor(seqlens, dtype=torch.int64), 0).to(torch.int32)
    hk, hv, d = case.hk, case.hv, case.d
    q = _bf16(torch.randn(t_tot, hk, d, generator=g))
    k = _bf16(torch.randn(t_tot, hk, d, generator=g))
    v = _bf16(torch.randn(t_tot, hv, d, generator=g))
    a = _bf16(torch.randn(t_tot, hv, generator=g))
    b = _bf16(torch.randn(t_tot, hv, generator=g))
    A_log = torch.log(torch.empty(hv).uniform_(1.0, 16.0, generator=g)).float()
    dt_bias = torch.randn(hv, generator=g).float()
    init_state = None
    if case.init_state:
        init_state = (torch.randn(n, hv, d, d, generator=g) * 0.1).float()
    z = w = None
    if case.gated_norm:
        z = _bf16(torch.randn(t_tot, hv, d, generator=g))
        w = _bf16(1.0 + 0.1 * torch.randn(d, generator=g))
    if case.a_log_const is not None:
        A_log = torch.full((hv,), float(case.a_log_const), dtype=torch.float32)
    if case.b_const is not None:
        b = _bf16(torch.full((t_tot, hv), float(case.b_const)))
    return dict(
        seqlens=seqlens, cu_seqlens=cu, q=q, k=k, v=v, a=a, b=b,
        A_log=A_log, dt_bias=dt_bias, init_state=init_state, z=z, norm_w=w,
        eps=case.eps, hk=hk, hv=hv, d=d,
    )


def make_decode_inputs(case: DecodeCase) -> dict:
    """Return CPU tensors for a decode case: persistent params + per-step tokens."""
    g = torch.Generator(device="cpu")
    g.manual_seed(case.seed)
    B, hk, hv, d = case.batch, case.hk, case.hv, case.d
    A_log = torch.log(torch.empty(hv).uniform_(1.0, 16.0, generator=g)).float()
    dt_bias = torch.randn(hv, generator=g).float()
    state = (torch.randn(B, hv, d, d, generator=g) * 0.1).float()
    steps = []
    for _ in range(case.steps):
        steps.append(dict(
            q=_bf16(torch.randn(B, hk, d, generator=g)),
            k=_bf16(torch.randn(B, hk, d, generator=g)),
            v=_bf16(torch.randn(B, hv, d, generator=g)),
            a=_bf16(torch.randn(B, hv, generator=g)),
            b=_bf16(torch.randn(B, hv, generator=g)),
        ))
    z = w = None
    if case.gated_norm:
        z = [_bf16(torch.randn(B, hv, d, generator=g)) for _ in range(case.steps)]
        w = _bf16(1.0 + 0.1 * torch.randn(d, generator=g))
    return dict(A_log=A_log, dt_bias=dt_bias, state=state, steps=steps, z=z,
                norm_w=w, eps=case.eps, hk=hk, hv=hv, d=d, batch=B)


def make_decode_slots_inputs(case: DecodeSlotsCase) -> dict:
    """Return CPU tensors for a slot-pool decode case.  Draw order: A_log,
    dt_bias, the pool, the slot permutation, the skipped and out-of-pool
    sequences, q, k, v, a, b, then z and w."""
    g = torch.Generator(device="cpu")
    g.manual_seed(case.seed)
    B, T, P, hk, hv, d = case.batch, case.tokens, case.slots, case.hk, case.hv, case.d
    A_log = torch.log(torch.empty(hv).uniform_(1.0, 16.0, generator=g)).float()
    dt_bias = torch.randn(hv, generator=g).float()
    pool = (torch.randn(P, hv, d, d, generator=g) * 0.1).float()
    idx = torch.randperm(P, generator=g)[:B].to(torch.int32)
    pick = torch.randperm(B, generator=g)
    idx[pick[:case.skipped]] = -1
    idx[pick[case.skipped:case.skipped + case.out_of_pool]] = P
    q = _bf16(torch.randn(B, T, hk, d, generator=g))
    k = _bf16(torch.randn(B, T, hk, d, generator=g))
    v = _bf16(torch.randn(B, T, hv, d, generator=g))
    a = _bf16(torch.randn(B, T, hv, generator=g))
    b = _bf16(torch.randn(B, T, hv, generator=g))
    z = w = None
    if case.gated_norm:
        z = _bf16(torch.randn(B, T, hv, d, generator=g))
        w = _bf16(1.0 + 0.1 * torch.randn(d, generator=g))
    return dict(q=q, k=k, v=v, a=a, b=b, A_log=A_log, dt_bias=dt_bias, pool=pool, state_idx=idx,
                z=z, norm_w=w, eps=case.eps, hk=hk, hv=hv, d=d, batch=B, tokens=T, slots=P)


def conv_channels(hk: int, hv: int, d: int = D_HEAD) -> int:
    """Channels of the short conv ahead of the core: q | k | v."""
    return (2 * hk + hv) * d


def make_conv_inputs(channels: int, width: int, rows: int, seed: int = 0, state: bool = True) -> dict:
    """Weights and carried states of the causal conv, from a generator of their
    own (so the core's inputs of a case do not change with the conv).  Draw
    order: weight [C, K] ~ U(-1/sqrt(K), 1/sqrt(K)) (the default fan-in bound
    of a depthwise conv), rounded to bf16; then, if ``state``, the carried raw
    inputs [rows, K-1, C] ~ N(0, 1) rounded to bf16, like the projections."""
    g = torch.Generator(device="cpu")
    g.manual_seed(10_000 + seed)
    bound = 1.0 / float(width) ** 0.5
    w = _bf16(torch.empty(channels, width).uniform_(-bound, bound, generator=g))
    st = _bf16(torch.randn(rows, width - 1, channels, generator=g)) if state else None
    return dict(weight=w, state=st, width=width, channels=channels)


# The workloads of the contract: the Qwen3.5-4B geometry (16/16/32/128) at
# T=64, 8x128 packed, T=2048 with the gated-RMSNorm epilogue, the Hv=48 varlen
# family member, and batch-256 decode over 64 steps.
CASE_T64 = PrefillCase("prefill_T64", seqlens=[64])
CASE_8x128 = PrefillCase("prefill_8x128_h0", seqlens=[128] * 8, init_state=True)
CASE_T2048 = PrefillCase("prefill_T2048_gnorm", seqlens=[2048], gated_norm=True)
CASE_VARLEN48 = PrefillCase("prefill_varlen16_hv48", n_random_seqs=16, hv=48, init_state=True)
CASE_DECODE = DecodeCase("decode_B256_64steps")


def to_f64(t: Optional[torch.Tensor]):
    """Exact upcast of a CPU tensor to a float64 numpy array (None passes through)."""
    if t is None:
        return None
    return t.to(torch.float64).numpy()
