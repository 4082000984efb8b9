"""Seeded synthetic KDA workloads shared by the tests, the smoke check and the
benchmark.

This module only draws random inputs with the distributions and shapes of the
workloads; it holds none of the method's arithmetic.  Both the CUDA path and
the fp64 oracle consume the tensors it returns (the oracle widens them to fp64
exactly, so both sides see the same values).

Distributions (per token and head):
  q, k  ~ N(0, 1), then L2-normalised over the key dimension
  v     ~ N(0, 1)
  beta  = sigmoid(N(0, 1))
  g     = -softplus(N(0, 1)) per key channel (log-decay, alpha = exp(g))
  gate  ~ N(0, 1);  norm weight w = 1 + N(0, 0.02);  eps = 1e-6
  initial pool states ~ N(0, 0.1)  (zero for the tiny workload)
Everything is drawn with ``torch.Generator`` on the CPU and rounded once to
the workload's dtype.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

__all__ = [
    "PrefillWorkload", "DecodeWorkload", "TINY", "VARLEN", "SCHED", "LONGPROMPT", "DECODE",
    "make_prefill", "make_decode_pool", "make_decode_step", "sched_lengths", "cu_from_lengths",
    "make_prefill_conv",
]


@dataclasses.dataclass(frozen=True)
class PrefillWorkload:
    name: str
    seqlens: tuple
    H: int
    dk: int
    dv: int
    chunk: int
    checkpoint_every: int
    in_dtype: torch.dtype
    state_dtype: torch.dtype
    num_slots: int
    gate: bool
    zero_state: bool
    seed: int
    slot_range: Optional[tuple] = None  # draw slots from [lo, hi); default whole pool

    @property
    def T(self) -> int:
        return int(sum(self.seqlens))

    @property
    def N(self) -> int:
        return len(self.seqlens)

    def replace(self, **kw) -> "PrefillWorkload":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    name: str
    N: int
    H: int
    dk: int
    dv: int
    in_dtype: torch.dtype
    state_dtype: torch.dtype
    num_slots: int
    gate: bool
    steps: int
    seed: int

    def replace(self, **kw) -> "DecodeWorkload":
        return dataclasses.replace(self, **kw)


def sched_lengths(total: int, parts: int, minimum: int, seed: int) -> tuple:
    """``parts`` lengths summing to ``total``, each >= ``minimum``: the minimum
    plus a uniform random composition of the rest (sorted uniform integer cut
    points)."""
    gen = torch.Generator().manual_seed(seed)
    rest = total - parts * minimum
    assert rest >= 0
    cuts = torch.randint(0, rest + 1, (parts - 1,), generator=gen).sort().values.tolist()
    edges = [0] + cuts + [rest]
    return tuple(minimum + edges[i + 1] - edges[i] for i in range(parts))


# Tiny prefill: 1 sequence, T=64, H=2, d=16, fp32 everywhere, chunk 16, zero state.
TINY = PrefillWorkload("tiny_T64_H2_d16_f32", (64,), 2, 16, 16, 16, 0, torch.float32,
                       torch.float32, 1, False, True, 0)
# Varlen prefill: lengths {37,128,200,512}, H=8, d=64, bf16 inputs, fp32 pool of 16.
VARLEN = PrefillWorkload("varlen_T877_H8_d64_bf16", (37, 128, 200, 512), 8, 64, 64, 64, 64,
                         torch.bfloat16, torch.float32, 16, False, False, 1)
# Scheduler step: 4096 tokens as 8 sequences (min 64), H=32, d=128, fp32 pool of
# 512 with slots from the top half, checkpoints every 256, fused norm-gate.
SCHED = PrefillWorkload("sched_T4096_N8_H32_d128_bf16", sched_lengths(4096, 8, 64, 2), 32, 128,
                        128, 64, 256, torch.bfloat16, torch.float32, 512, True, False, 2,
                        slot_range=(256, 512))
# Long prompt: one 32768-token sequence (run as 8 calls of 4096), bf16 state.
LONGPROMPT = PrefillWorkload("longprompt_T32768_H32_d128_bf16state", (32768,), 32, 128, 128, 64,
                             256, torch.bfloat16, torch.bfloat16, 8, False, False, 3)
# Recurrent decode: 256 sequences x 1 token, H=32, d=128, fp32 pool of 1024, 64 steps.
DECODE = DecodeWorkload("decode_N256_H32_d128_pool1024", 256, 32, 128, 128, torch.bfloat16,
                        torch.float32, 1024, True, 64, 4)


def cu_from_lengths(lengths: Sequence[int]) -> torch.Tensor:
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32)


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)


def _token_inputs(gen, T, H, dk, dv, dtype, gate):
    q = _unit_rows(torch.randn(T, H, dk, generator=gen, dtype=torch.float64))
    k = _unit_rows(torch.randn(T, H, dk, generator=gen, dtype=torch.float64))
    v = torch.randn(T, H, dv, generator=gen, dtype=torch.float64)
    g = -torch.nn.functional.softplus(torch.randn(T, H, dk, generator=gen, dtype=torch.float64))
    beta = torch.sigmoid(torch.randn(T, H, generator=gen, dtype=torch.float64))
    out = dict(q=q.to(dtype), k=k.to(dtype), v=v.to(dtype), g=g.to(dtype), beta=beta.to(dtype))
    if gate:
        out["gate"] = torch.randn(T, H, dv, generator=gen, dtype=torch.float64).to(dtype)
    return out


def _norm_weight(gen, dv, dtype):
    return (1.0 + 0.02 * torch.randn(dv, generator=gen, dtype=torch.float64)).to(dtype)


def _pool(gen, num_slots, H, dk, dv, dtype, zero):
    if zero:
        return torch.zeros(num_slots, H, dk, dv, dtype=dtype)
    # Drawn in fp32 to keep large pools cheap to generate.
    return (0.1 * torch.randn(num_slots, H, dk, dv, generator=gen, dtype=torch.float32)).to(dtype)


def _slots(gen, n, num_slots, slot_range=None):
    lo, hi = slot_range if slot_range else (0, num_slots)
    assert hi - lo >= n
    return (lo + torch.randperm(hi - lo, generator=gen)[:n]).to(torch.int32)


def make_prefill(w: PrefillWorkload, *, lengths: Optional[Sequence[int]] = None, seed=None):
    """Inputs for one prefill call of workload ``w`` (CPU tensors).

    Returns a dict with q,k,v,g,beta [T,H,*] in ``w.in_dtype``, cu_seqlens and
    state_indices (int32), pool [num_slots,H,dk,dv] in ``w.state_dtype``,
    gate/norm_w (or None), eps and scale.
    """
    lengths = tuple(lengths) if lengths is not None else w.seqlens
    seed = w.seed if seed is None else seed
    gen = torch.Generator().manual_seed(int(seed))
    T = int(sum(lengths))
    d = _token_inputs(gen, T, w.H, w.dk, w.dv, w.in_dtype, w.gate)
    d["norm_w"] = _norm_weight(gen, w.dv, w.in_dtype) if w.gate else None
    d.setdefault("gate", None)
    d["state_indices"] = _slots(gen, len(lengths), w.num_slots, w.slot_range)
    d["pool"] = _pool(gen, w.num_slots, w.H, w.dk, w.dv, w.state_dtype, w.zero_state)
    d["cu_seqlens"] = cu_from_lengths(lengths)
    d["eps"] = 1e-6
    d["scale"] = 1.0 / math.sqrt(w.dk)
    return d


def make_prefill_conv(w: PrefillWorkload, conv_width: int, *, lengths: Optional[Sequence[int]] = None,
                      seed=None):
    """Inputs of the prefill with the short convolution in front: those of
    make_prefill without q, k, v (the convolution makes them), plus the packed
    projection x [T, 3*H*dk] ~ N(0, 1) (channels q, then k, then v), taps
    conv_w [3*H*dk, W] ~ N(0, 0.5^2), bias conv_b [3*H*dk] ~ N(0, 0.1^2) and a
    convolution cache pool conv_pool [num_slots, W-1, 3*H*dk] ~ N(0, 1), all
    in ``w.in_dtype``."""
    d = make_prefill(w, lengths=lengths, seed=seed)
    for key in ("q", "k", "v"):
        d.pop(key)
    gen = torch.Generator().manual_seed(int(w.seed if seed is None else seed) + 7919)
    C3 = 3 * w.H * w.dk
    T = int(d["cu_seqlens"][-1])
    d["x"] = torch.randn(T, C3, generator=gen, dtype=torch.float32).to(w.in_dtype)
    d["conv_w"] = (0.5 * torch.randn(C3, conv_width, generator=gen, dtype=torch.float32)).to(w.in_dtype)
    d["conv_b"] = (0.1 * torch.randn(C3, generator=gen, dtype=torch.float32)).to(w.in_dtype)
    d["conv_pool"] = torch.randn(w.num_slots, conv_width - 1, C3, generator=gen,
                                 dtype=torch.float32).to(w.in_dtype)
    return d


def make_prefill_segment(w: PrefillWorkload, lengths: Sequence[int], seed: int):
    """Token inputs only (q,k,v,g,beta[,gate]) for a continuation segment."""
    gen = torch.Generator().manual_seed(int(seed))
    return _token_inputs(gen, int(sum(lengths)), w.H, w.dk, w.dv, w.in_dtype, w.gate)


def make_decode_pool(w: DecodeWorkload, seed=None):
    """Pool, slot indices and norm weight for a decode workload."""
    gen = torch.Generator().manual_seed(int(w.seed if seed is None else seed))
    pool = _pool(gen, w.num_slots, w.H, w.dk, w.dv, w.state_dtype, False)
    idx = _slots(gen, w.N, w.num_slots)
    norm_w = _norm_weight(gen, w.dv, w.in_dtype) if w.gate else None
    return dict(pool=pool, state_indices=idx, norm_w=norm_w, eps=1e-6,
                scale=1.0 / math.sqrt(w.dk))


def make_decode_step(w: DecodeWorkload, step: int, seed=None):
    """Fresh per-step token inputs (q,k,v,g,beta[,gate]) of shape [N,H,*]."""
    base = w.seed if seed is None else seed
    gen = torch.Generator().manual_seed(int(base) * 1_000_003 + 7919 * (step + 1))
    return _token_inputs(gen, w.N, w.H, w.dk, w.dv, w.in_dtype, w.gate)



def make_decode_draft(w: DecodeWorkload, K: int, seed=None):
    """Inputs of K draft tokens per sequence for speculative-decoding
    verification: q,k,g [N,K,H,dk]; v, gate [N,K,H,dv]; beta [N,K,H]; the
    accepted-prefix lengths a_i, uniform in [0, K]."""
    base = w.seed if seed is None else seed
    gen = torch.Generator().manual_seed(int(base) * 1_000_003 + 104729 * K)
    t = _token_inputs(gen, w.N * K, w.H, w.dk, w.dv, w.in_dtype, w.gate)
    out = {name: x.reshape((w.N, K) + tuple(x.shape[1:])) for name, x in t.items()}
    out["num_accepted"] = torch.randint(0, K + 1, (w.N,), generator=gen, dtype=torch.int32)
    return out


def make_conv(lengths, C: int, W: int, dtype, num_slots: int, seed: int, has_initial=None):
    """Inputs of the short causal convolution: x [T, C] ~ N(0, 1) (the
    projections), taps [C, W] ~ N(0, 0.5^2), bias [C] ~ N(0, 0.1^2), cache pool
    [num_slots, W-1, C] ~ N(0, 1), distinct slots from a seeded permutation."""
    gen = torch.Generator().manual_seed(int(seed))
    T = int(sum(lengths))
    x = torch.randn(T, C, generator=gen, dtype=torch.float64).to(dtype)
    w = (0.5 * torch.randn(C, W, generator=gen, dtype=torch.float64)).to(dtype)
    b = (0.1 * torch.randn(C, generator=gen, dtype=torch.float64)).to(dtype)
    pool = torch.randn(num_slots, W - 1, C, generator=gen, dtype=torch.float32).to(dtype)
    idx = _slots(gen, len(lengths), num_slots)
    out = dict(x=x, w=w, b=b, pool=pool, state_indices=idx, cu_seqlens=cu_from_lengths(lengths))
    if has_initial is not None:
        out["has_initial_state"] = torch.tensor(has_initial, dtype=torch.int32)
    return out
