"""Helpers shared by the GPU parity tests: device transfer, the oracle call on
the same inputs, and the tolerance rule.

Tolerance rule.  The bound is max-abs 0.01 when the state is fp32 and 0.03
when it is bf16 (the FlashKDA checkpoint test's tolerances).  Values the ABI
stores in bf16 or fp16 (outputs with 16-bit inputs, bf16 states) carry an
unavoidable final rounding of half an ulp; that rounding is allowed on top of
the bound: |gpu - oracle| <= tol + ulp_half(oracle).
"""
from __future__ import annotations

import numpy as np
import torch


def tol_for(state_dtype) -> float:
    return 0.03 if state_dtype == torch.bfloat16 else 0.01


def half_ulp(ref: np.ndarray, dtype) -> np.ndarray:
    """Half a unit in the last place of ref in the stored dtype (bf16: 8
    significant bits, fp16: 11; fp32 results get no allowance)."""
    bits = {torch.bfloat16: 8, torch.float16: 11}.get(dtype)
    if bits is None:
        return np.zeros_like(ref)
    a = np.abs(ref)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    if dtype == torch.float16:
        e = np.maximum(e, -14.0)  # subnormal spacing
    return np.where(a > 0, 2.0 ** (e - bits), 0.0)


def excess_error(gpu: torch.Tensor, ref: np.ndarray) -> float:
    """max(|gpu - ref| - half_ulp(ref)) in fp64 (<= tol means within bounds)."""
    g = gpu.detach().double().cpu().numpy()
    if g.size == 0:
        return 0.0
    return float(np.max(np.abs(g - ref) - half_ulp(ref, gpu.dtype)))


# Errors measured by the parity tests of the named workloads, written out at
# the end of the session when KDA_PARITY_REPORT names a file (conftest).
PARITY_ERRORS: dict = {}


def record(workload: str, what: str, gpu: torch.Tensor, ref: np.ndarray) -> None:
    """Keep the raw max-abs error and its excess over the half-ulp allowance
    for one compared quantity of a named workload (the worst over calls)."""
    g = gpu.detach().double().cpu().numpy()
    if g.size == 0:
        return
    raw = float(np.max(np.abs(g - ref)))
    exc = float(np.max(np.abs(g - ref) - half_ulp(ref, gpu.dtype)))
    ent = PARITY_ERRORS.setdefault(workload, {}).setdefault(what, {"raw_max_abs": 0.0,
                                                                   "excess_over_half_ulp": -1e30})
    ent["raw_max_abs"] = max(ent["raw_max_abs"], raw)
    ent["excess_over_half_ulp"] = max(ent["excess_over_half_ulp"], exc)


def max_abs(gpu: torch.Tensor, ref: np.ndarray) -> float:
    g = gpu.detach().double().cpu().numpy()
    return float(np.max(np.abs(g - ref))) if g.size else 0.0


def to_dev(d: dict, dev) -> dict:
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def run_prefill(kda, d, w, dev, *, lengths=None, ckpt=True, out_dtype=None):
    """Run kda_prefill_chunked on inputs ``d`` (CPU tensors); returns the
    device tensors (out, pool, checkpoints, offsets, status)."""
    t = to_dev(d, dev)
    T = t["q"].shape[0]
    N = t["state_indices"].shape[0]
    I = w.checkpoint_every if ckpt else 0
    cap = max(T // I, 1) if I else 0
    ck = torch.full((cap, w.H, w.dk, w.dv), float("nan"), device=dev,
                    dtype=w.state_dtype) if I else None
    offs = torch.full((N + 1,), -7, dtype=torch.int32, device=dev)
    out = torch.full((T, w.H, w.dv), float("nan"), device=dev, dtype=w.in_dtype)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws_bytes = kda.kda_prefill_workspace_bytes(N, T, w.H, w.dk, w.dv, w.chunk)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev) if ws_bytes else None
    kda.kda_prefill_chunked(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"],
                            t["state_indices"], t["pool"], out, chunk=w.chunk, checkpoints=ck,
                            checkpoint_every=I, ckpt_offsets=offs, gate=t.get("gate"),
                            norm_w=t.get("norm_w"), eps=d.get("eps", 1e-6), scale=d["scale"],
                            gate_act=d.get("gate_act", "sigmoid"),
                            has_initial_state=t.get("has_initial_state"), workspace=ws,
                            dev_status=status)
    torch.cuda.synchronize()
    return out, t["pool"], ck, offs, status


def oracle_prefill(oracle, d, w, *, ckpt=True, heads=None):
    """The fp64 oracle on the same inputs; ``heads`` restricts to a subset."""
    sel = (lambda x: x) if heads is None else (lambda x: x[:, heads])
    psel = (lambda x: x) if heads is None else (lambda x: x[:, heads])
    gate = d.get("gate")
    return oracle.prefill(sel(d["q"]), sel(d["k"]), sel(d["v"]), sel(d["g"]), sel(d["beta"]),
                          d["cu_seqlens"], d["state_indices"], psel(d["pool"]),
                          checkpoint_every=w.checkpoint_every if ckpt else 0,
                          gate=None if gate is None else sel(gate), norm_w=d.get("norm_w"),
                          eps=d.get("eps", 1e-6), scale=d["scale"],
                          gate_act=d.get("gate_act", "sigmoid"),
                          has_initial_state=d.get("has_initial_state"))


def run_prefill_conv(kda, d, w, dev, *, conv_act="silu", ckpt=True):
    """Run kda_prefill_chunked_conv on inputs ``d`` (CPU tensors, from
    make_prefill_conv); returns the device tensors (out, pool, checkpoints,
    offsets, status, conv_pool)."""
    t = to_dev(d, dev)
    T = t["x"].shape[0]
    N = t["state_indices"].shape[0]
    I = w.checkpoint_every if ckpt else 0
    cap = max(T // I, 1) if I else 0
    ck = torch.full((cap, w.H, w.dk, w.dv), float("nan"), device=dev,
                    dtype=w.state_dtype) if I else None
    offs = torch.full((N + 1,), -7, dtype=torch.int32, device=dev)
    out = torch.full((T, w.H, w.dv), float("nan"), device=dev, dtype=w.in_dtype)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws_bytes = kda.kda_prefill_workspace_bytes(N, T, w.H, w.dk, w.dv, w.chunk)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev) if ws_bytes else None
    kda.kda_prefill_chunked_conv(t["x"], t["conv_w"], t["conv_pool"], t["g"], t["beta"], t["cu_seqlens"],
                                 t["state_indices"], t["pool"], out, conv_b=t.get("conv_b"),
                                 conv_act=conv_act, chunk=w.chunk, checkpoints=ck, checkpoint_every=I,
                                 ckpt_offsets=offs, gate=t.get("gate"), norm_w=t.get("norm_w"),
                                 eps=d.get("eps", 1e-6), scale=d["scale"],
                                 gate_act=d.get("gate_act", "sigmoid"),
                                 has_initial_state=t.get("has_initial_state"), workspace=ws,
                                 dev_status=status)
    torch.cuda.synchronize()
    return out, t["pool"], ck, offs, status, t["conv_pool"]


def oracle_prefill_conv(oracle, d, w, *, conv_act="silu", ckpt=True):
    """oracle.prefill_conv on the same inputs, with every stage's result
    stored in the inputs' dtype."""
    T = d["x"].shape[0]
    x = d["x"].reshape(T, 3, w.H, w.dk)
    return oracle.prefill_conv(x[:, 0], x[:, 1], x[:, 2], d["conv_w"], d["cu_seqlens"], d["state_indices"],
                               d["pool"], d["conv_pool"], conv_bias=d.get("conv_b"), conv_act=conv_act,
                               has_initial_state=d.get("has_initial_state"), dtype=w.in_dtype,
                               g=d["g"], beta=d["beta"],
                               checkpoint_every=w.checkpoint_every if ckpt else 0, gate=d.get("gate"),
                               norm_w=d.get("norm_w"), eps=d.get("eps", 1e-6), scale=d["scale"],
                               gate_act=d.get("gate_act", "sigmoid"))
