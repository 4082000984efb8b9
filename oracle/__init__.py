"""fp64 CPU oracle for Kimi Delta Attention -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The CUDA library never links or calls it, and it shares
no code with it.

The arithmetic lives in ``kda_oracle.c`` (plain C, fp64, token by token); this
module compiles it with gcc on first use and marshals numpy arrays through
ctypes.  See the C file's header for what is computed and which page passage
each part follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None

ERRORS = {0: "ok", -1: "invalid argument", -2: "state index out of range",
          -3: "checkpoint capacity too small", -4: "out of memory"}


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libkda_oracle.so``."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            lib.kda_oracle_prefill.restype = ctypes.c_int
            lib.kda_oracle_prefill.argtypes = [
                P, P, P, P, P, P, ctypes.c_int, P, P, P, ctypes.c_int64, P, P, ctypes.c_int,
                ctypes.c_int64, P, P, P, ctypes.c_double, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int]
            lib.kda_oracle_decode.restype = ctypes.c_int
            lib.kda_oracle_decode.argtypes = [
                P, P, P, P, P, P, ctypes.c_int, P, ctypes.c_int64, P, P, P, ctypes.c_double,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                ctypes.c_int]
            lib.kda_oracle_norm_gate.restype = ctypes.c_int
            lib.kda_oracle_norm_gate.argtypes = [P, P, P, ctypes.c_double, P, ctypes.c_int64,
                                                 ctypes.c_int, ctypes.c_int]
            lib.kda_oracle_norm_gate_ex.restype = ctypes.c_int
            lib.kda_oracle_norm_gate_ex.argtypes = [P, P, P, ctypes.c_int64, P, P, ctypes.c_double,
                                                    ctypes.c_int, P, P, ctypes.c_int64, ctypes.c_int,
                                                    ctypes.c_int]
            lib.kda_oracle_conv_prefill.restype = ctypes.c_int
            lib.kda_oracle_conv_prefill.argtypes = [P, P, P, P, ctypes.c_int, P, P, P, ctypes.c_int64,
                                                    ctypes.c_int, ctypes.c_int, ctypes.c_int, P]
            lib.kda_oracle_checkpoint_offsets.restype = ctypes.c_int64
            lib.kda_oracle_checkpoint_offsets.argtypes = [P, ctypes.c_int, ctypes.c_int, P]
            lib.kda_oracle_max_threads.restype = ctypes.c_int
            lib.kda_oracle_max_threads.argtypes = []
            _lib = lib
    return _lib


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # a torch tensor: widen exactly on the CPU
        a = a.detach().cpu().double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a):
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc):
    if rc != 0:
        raise OracleError(ERRORS.get(rc, f"error {rc}"))


def max_threads() -> int:
    return _load().kda_oracle_max_threads()


def checkpoint_offsets(cu_seqlens, every: int) -> np.ndarray:
    """Exclusive prefix sum of floor(len_i / every) over the sequences ([N+1])."""
    cu = _i32(cu_seqlens)
    n = cu.shape[0] - 1
    offs = np.zeros(n + 1, np.int32)
    total = _load().kda_oracle_checkpoint_offsets(_ptr(cu), n, int(every), _ptr(offs))
    if total < 0:
        raise OracleError("malformed cu_seqlens")
    return offs


ACT = {"sigmoid": 0, "silu": 1}


def prefill(q, k, v, g, beta, cu_seqlens, state_indices, pool, *, checkpoint_every=0,
            gate=None, norm_w=None, eps=1e-6, scale=None, nthreads=0, has_initial_state=None,
            gate_act="sigmoid"):
    """Token-by-token KDA prefill in fp64.

    Shapes: q,k,g [T,H,dk]; v [T,H,dv]; beta [T,H]; cu_seqlens [N+1];
    state_indices [N]; pool [num_slots,H,dk,dv].  Returns
    ``(out [T,H,dv], pool_after [num_slots,H,dk,dv], checkpoints [n,H,dk,dv],
    ckpt_offsets [N+1])``.  The input pool is not modified.
    """
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    cu, idx = _i32(cu_seqlens), _i32(state_indices)
    his = None if has_initial_state is None else _i32(has_initial_state)
    pool = _f64(pool).copy()
    gate, norm_w = _f64(gate), _f64(norm_w)
    T, H, dk = q.shape
    dv = v.shape[-1]
    N = idx.shape[0]
    if scale is None or scale <= 0:
        scale = 1.0 / np.sqrt(dk)
    offs = checkpoint_offsets(cu, checkpoint_every) if N > 0 else np.zeros(1, np.int32)
    n_ck = int(offs[-1])
    ck = np.zeros((max(n_ck, 1), H, dk, dv), np.float64)
    out = np.zeros((T, H, dv), np.float64)
    offs_out = np.zeros(N + 1, np.int32)
    rc = _load().kda_oracle_prefill(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu), N, _ptr(idx), _ptr(his),
        _ptr(pool), pool.shape[0], _ptr(out), _ptr(ck), int(checkpoint_every), ck.shape[0],
        _ptr(offs_out), _ptr(gate), _ptr(norm_w), float(eps), ACT[gate_act], H, dk, dv,
        float(scale), int(nthreads))
    _check(rc)
    return out, pool, ck[:n_ck], offs_out


def decode(q, k, v, g, beta, state_indices, pool, *, gate=None, norm_w=None, eps=1e-6,
           scale=None, nthreads=0, gate_act="sigmoid"):
    """One recurrent decode step in fp64.  q,k,g [N,H,dk]; v [N,H,dv]; beta [N,H].

    Returns ``(out [N,H,dv], pool_after)``; the input pool is not modified.
    """
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    idx = _i32(state_indices)
    pool = _f64(pool).copy()
    gate, norm_w = _f64(gate), _f64(norm_w)
    N, H, dk = q.shape
    dv = v.shape[-1]
    if scale is None or scale <= 0:
        scale = 1.0 / np.sqrt(dk)
    out = np.zeros((N, H, dv), np.float64)
    rc = _load().kda_oracle_decode(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(idx), N, _ptr(pool), pool.shape[0],
        _ptr(out), _ptr(gate), _ptr(norm_w), float(eps), ACT[gate_act], H, dk, dv, float(scale),
        int(nthreads))
    _check(rc)
    return out, pool


def decode_multi(q, k, v, g, beta, state_indices, pool, *, gate=None, norm_w=None, eps=1e-6,
                 scale=None, nthreads=0, gate_act="sigmoid"):
    """K recurrent decode steps per sequence, keeping the state after each token
    (speculative-decoding verification: "[Feature][KDA] Add Kimi K3 KDA
    execution", section "Metadata construction", and the FlashKDA summary's
    risk section).  Each step is :func:`decode` on the pool left by the previous
    one.  q,k,g [N,K,H,dk]; v, gate [N,K,H,dv]; beta [N,K,H].

    Returns ``(out [N,K,H,dv], token_states [N,K,H,dk,dv], pool_after_K)``;
    token_states rows of padding sequences (index -1) are NaN.
    """
    q, k, v, g, beta, gate = (_f64(x) for x in (q, k, v, g, beta, gate))
    N, K, H, dk = q.shape
    dv = v.shape[-1]
    idx = _i32(state_indices)
    cur = _f64(pool).copy()
    out = np.zeros((N, K, H, dv), np.float64)
    states = np.full((N, K, H, dk, dv), np.nan)
    live = idx >= 0
    for t in range(K):
        out[:, t], cur = decode(q[:, t], k[:, t], v[:, t], g[:, t], beta[:, t], idx, cur,
                                gate=None if gate is None else gate[:, t],
                                norm_w=norm_w, eps=eps, scale=scale, nthreads=nthreads,
                                gate_act=gate_act)
        states[live, t] = cur[idx[live]]
    return out, states, cur


def commit_accepted(token_states, num_accepted, state_indices, pool):
    """pool[idx_i] = token_states[i, a_i - 1] for a_i = num_accepted[i] >= 1;
    a_i == 0 or idx_i == -1 leaves the slot unchanged."""
    pool = _f64(pool).copy()
    token_states = _f64(token_states)
    for i, (slot, a) in enumerate(zip(_i32(state_indices), _i32(num_accepted))):
        if slot >= 0 and a >= 1:
            pool[slot] = token_states[i, a - 1]
    return pool


def norm_gate(o, gate, w, eps=1e-6, gate_act="sigmoid"):
    """y = o / sqrt(mean(o^2)+eps) * w * act(gate) over the last dimension."""
    o, gate, w = _f64(o), _f64(gate), _f64(w)
    dv = o.shape[-1]
    rows = o.size // dv
    y = np.zeros_like(o)
    _check(_load().kda_oracle_norm_gate(_ptr(o), _ptr(gate), _ptr(w), float(eps), _ptr(y),
                                        rows, dv, ACT[gate_act]))
    return y


def norm_gate_ex(o, gate, *, residual=None, w=None, b=None, eps=1e-6, gate_act="sigmoid",
                 gate_row_stride=0):
    """Norm-gate variants: x = o + residual; z = x / sqrt(mean(x^2)+eps) * w + b;
    y = z * act(gate).  o, residual: [rows, H, dv]; gate: flat buffer whose row r
    (all heads) starts at r * gate_row_stride (0: H*dv, i.e. [rows, H, dv]).
    Returns ``(y, residual_out)``, residual_out = x."""
    o = _f64(o)
    rows, H, dv = o.shape
    residual, w, b = _f64(residual), _f64(w), _f64(b)
    gate = _f64(gate).reshape(-1)
    stride = gate_row_stride or H * dv
    y = np.zeros_like(o)
    res_out = np.zeros_like(o)
    _check(_load().kda_oracle_norm_gate_ex(_ptr(o), _ptr(residual), _ptr(gate), int(stride), _ptr(w),
                                           _ptr(b), float(eps), ACT[gate_act], _ptr(y), _ptr(res_out),
                                           rows, H, dv))
    return y, res_out


CONV_ACT = {"none": 0, "silu": 1}


def conv_prefill(x, w, cu_seqlens, state_indices, pool, *, bias=None, has_initial_state=None,
                 act="silu"):
    """Short causal convolution over packed sequences ("[Feature][KDA] Add Kimi
    K3 KDA execution", "KDA execution" step 2).  x [T, C]; w [C, W]; bias [C];
    pool [slots, W-1, C].  Returns ``(y [T, C], pool_after)``; the input pool is
    not modified."""
    x, w, bias = _f64(x), _f64(w), _f64(bias)
    pool = _f64(pool).copy()
    cu, idx = _i32(cu_seqlens), _i32(state_indices)
    his = None if has_initial_state is None else _i32(has_initial_state)
    T, C = x.shape
    W = w.shape[1]
    y = np.zeros((T, C), np.float64)
    _check(_load().kda_oracle_conv_prefill(_ptr(x), _ptr(w), _ptr(bias), _ptr(cu), len(idx), _ptr(idx),
                                           _ptr(his), _ptr(pool), pool.shape[0], C, W,
                                           CONV_ACT[act], _ptr(y)))
    return y, pool


def conv_decode(x, w, state_indices, pool, *, bias=None, act="silu"):
    """One token per sequence: the prefill of a length-1 segment per sequence
    (the cache supplies the W-1 earlier inputs).  x [N, C]."""
    x = _f64(x)
    N = x.shape[0]
    cu = np.arange(N + 1, dtype=np.int32)
    return conv_prefill(x, w, cu, state_indices, pool, bias=bias, act=act)


def l2_normalize(x, eps=1e-6):
    """Rows of unit L2 norm over the last axis: x / sqrt(sum(x^2) + eps), in
    fp64.  The pages apply the short convolution to Q/K/V and then run the
    chunk prefill ("[Feature][KDA] Add Kimi K3 KDA execution", "KDA
    execution" steps 2-3); the recurrence's regime is q and k rows of unit
    norm, so the composed operator normalises q and k per (token, head) in
    between (the eps keeps a zero row at zero)."""
    x = _f64(x)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def _stored(x, dtype):
    """``x`` as a tensor of ``dtype`` would hold it (round to nearest even),
    widened back to fp64: the value a stage of the pipeline hands to the next
    through a tensor of that dtype."""
    import torch
    return torch.from_numpy(_f64(x)).to(dtype).double().numpy()


def prefill_conv(xq, xk, xv, conv_w, cu_seqlens, state_indices, pool, conv_pool, *, conv_bias=None,
                 conv_act="silu", has_initial_state=None, dtype=None, l2_eps=1e-6, **prefill_kw):
    """The convolution, the normalisation and the chunk prefill as the pages'
    pipeline runs them, each stage reading the previous one's output tensor:

      q, k, v = act(conv(x)) over the packed channels [q | k | v] of each
                token, with the convolution cache of state_indices[i]
                (conv_prefill), stored in ``dtype``;
      q, k    = l2_normalize per (token, head), stored in ``dtype``;
      the chunked prefill (prefill) on q, k, v and the caller's g, beta.

    xq, xk, xv [T, H, d]; conv_w [3*H*d, W] (channels q, then k, then v, head
    by head); conv_pool [slots, W-1, 3*H*d].  ``dtype`` (a torch dtype, or None
    for no rounding) is the activation dtype.  Returns ``(out, pool_after,
    checkpoints, ckpt_offsets, conv_pool_after)``."""
    xq, xk, xv = _f64(xq), _f64(xk), _f64(xv)
    T, H, d = xq.shape
    x = np.concatenate([xq.reshape(T, H * d), xk.reshape(T, H * d), xv.reshape(T, H * d)], axis=1)
    y, conv_after = conv_prefill(x, conv_w, cu_seqlens, state_indices, conv_pool, bias=conv_bias,
                                 has_initial_state=has_initial_state, act=conv_act)
    rnd = (lambda a: a) if dtype is None else (lambda a: _stored(a, dtype))
    y = rnd(y)
    q, k, v = (y[:, i * H * d:(i + 1) * H * d].reshape(T, H, d) for i in range(3))
    q, k = rnd(l2_normalize(q, l2_eps)), rnd(l2_normalize(k, l2_eps))
    out, pool_after, ck, offs = prefill(q, k, v, prefill_kw.pop("g"), prefill_kw.pop("beta"), cu_seqlens,
                                        state_indices, pool, has_initial_state=has_initial_state,
                                        **prefill_kw)
    return out, pool_after, ck, offs, conv_after
