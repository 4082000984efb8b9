"""Python binding of libkda (KDA prefill, decode and output norm-gate on GB300).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libkda.so``; torch supplies device memory and streams.  Each
function carries the C entry point's name and passes torch tensors as raw
pointers.  There is no fallback: if ``libkda.so`` is missing or fails to load,
every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

__all__ = [
    "load", "lib_path", "KdaError", "KDA_OK", "KDA_F32", "KDA_BF16",
    "kda_prefill_chunked", "kda_prefill_workspace_bytes", "kda_decode_step", "kda_norm_gate",
    "kda_status_string", "kda_version", "DEV_STATUS", "prefill_launches",
    "kda_prefill_chunked_static_scratch", "STATIC_SCRATCH_BYTES", "kda_decode_multi",
    "kda_commit_accepted", "kda_norm_gate_ex", "KDA_F16", "kda_causal_conv1d_prefill",
    "kda_causal_conv1d_decode", "kda_testing_set_first_wait_tries", "kda_prefill_path",
    "kda_prefill_chunked_conv",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libkda.so")
_lib = None

KDA_OK, KDA_F32, KDA_BF16, KDA_F16 = 0, 0, 1, 2
GATE_ACT = {"sigmoid": 0, "silu": 1}  # kda_gate_act
STATIC_SCRATCH_BYTES = 128 << 20  # KDA_STATIC_SCRATCH_BYTES in include/kda.h
DEV_STATUS = {0: "ok", 1: "bad state index", 2: "bad cu_seqlens", 3: "on-chip wait timeout",
              4: "checkpoint capacity exceeded", 5: "state slot named twice in one call"}

_P = ctypes.c_void_p
_I32, _I64, _F32, _SZ = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t

_SIGNATURES = {
    "kda_prefill_workspace_bytes": (_SZ, [ctypes.c_int, _I64, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int]),
    "kda_prefill_chunked": (ctypes.c_int, [
        _P, _P, _P, _P, _P, ctypes.c_int, _P, ctypes.c_int, _I64, _P, _P, _P, _I64, ctypes.c_int,
        _P, _P, _I32, _I64, _P, _P, _P, _F32, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_int, _F32, _P, _SZ, _P, _P]),
    "kda_decode_step": (ctypes.c_int, [
        _P, _P, _P, _P, _P, ctypes.c_int, _P, ctypes.c_int, _P, _I64, ctypes.c_int, _P, _P, _P,
        _F32, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _F32, _P, _P]),
    "kda_decode_multi": (ctypes.c_int, [
        _P, _P, _P, _P, _P, ctypes.c_int, _P, ctypes.c_int, ctypes.c_int, _P, _I64, ctypes.c_int,
        _P, _P, ctypes.c_int, _P, _P, _F32, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        _F32, _P, _P]),
    "kda_commit_accepted": (ctypes.c_int, [
        _P, _P, _P, ctypes.c_int, ctypes.c_int, _P, _I64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, _P, _P]),
    "kda_causal_conv1d_prefill": (ctypes.c_int, [
        _P, _P, _P, ctypes.c_int, _P, ctypes.c_int, _I64, ctypes.c_int, ctypes.c_int, _P, _P, _P,
        _I64, ctypes.c_int, _P, _P, _P]),
    "kda_causal_conv1d_decode": (ctypes.c_int, [
        _P, _P, _P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P, _I64, ctypes.c_int,
        _P, _P, _P]),
    "kda_norm_gate_ex": (ctypes.c_int, [_P, _P, _P, _P, _I64, _P, _P, _F32, ctypes.c_int, _P, _I64,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int, _P]),
    "kda_norm_gate": (ctypes.c_int, [_P, _P, _P, _F32, ctypes.c_int, _P, _I64, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_int, _P]),
    "kda_prefill_chunked_static_scratch": (ctypes.c_int, [
        _P, _P, _P, _P, _P, ctypes.c_int, _P, ctypes.c_int, _I64, _P, _P, _P, _I64, ctypes.c_int,
        _P, _P, _I32, _I64, _P, _P, _P, _F32, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_int, _F32, _P, _P]),
    "kda_prefill_chunked_conv": (ctypes.c_int, [
        _P, _P, _P, _I64, _P, _P, ctypes.c_int, ctypes.c_int, _P, _I64,
        _P, _P, ctypes.c_int, _P, ctypes.c_int, _I64, _P, _P, _P, _I64, ctypes.c_int,
        _P, _P, _I32, _I64, _P, _P, _P, _F32, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_int, _F32, _P, _SZ, _P, _P]),
    "kda_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "kda_testing_set_first_wait_tries": (None, [_I32, _I32]),
    "kda_prefill_path": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "kda_version": (ctypes.c_int, []),
}


class KdaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {kda_status_string(status)} ({status})")


def lib_path() -> str:
    return _LIB_PATH


def load():
    """Load libkda.so (built by ``build.py``); raises when it is absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libkda.so not built ({_LIB_PATH}); run the package's build.py")
        lib = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype, fn.argtypes = res, args
        _lib = lib
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("libkda takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr()) if t.numel() > 0 else None


def _need(t, name, shape=None, dtype=None, device=None):
    """Raise ValueError unless ``t`` (when given) is a CUDA tensor on ``device``
    (the device of the call's first tensor), of ``shape`` (None entries match
    any size) and ``dtype``.  The C ABI takes bare device pointers and launches
    on the current device, so a host tensor, a tensor on another GPU, a
    mismatched size or an int64 index array would otherwise be read as
    something it is not."""
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device} but the call's tensors are on {device}: "
                         "every tensor of a call must be on one CUDA device")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if shape is not None and (t.dim() != len(shape) or any(
            s is not None and int(a) != int(s) for a, s in zip(t.shape, shape))):
        want = tuple("*" if s is None else int(s) for s in shape)
        raise ValueError(f"{name} must have shape {want}, got {tuple(t.shape)}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _one_device(dev, **tensors):
    """Raise ValueError unless every given tensor is on ``dev``; runs before
    the per-tensor checks so that a mixed call is named as such."""
    for name, t in tensors.items():
        if isinstance(t, torch.Tensor) and t.device != dev:
            raise ValueError(f"{name} is on {t.device} but the call's tensors are on {dev}: "
                             "every tensor of a call must be on one CUDA device")


def _need_prefill(q, k, v, g, beta, cu_seqlens, state_indices, state_pool, out, checkpoints,
                  ckpt_offsets, gate, norm_w, has_initial_state, dev_status):
    T, H, dk = q.shape
    dv = v.shape[-1]
    dev = q.device
    _one_device(dev, k=k, v=v, g=g, beta=beta, cu_seqlens=cu_seqlens, state_indices=state_indices,
                state_pool=state_pool, out=out, checkpoints=checkpoints, ckpt_offsets=ckpt_offsets,
                gate=gate, norm_w=norm_w, has_initial_state=has_initial_state, dev_status=dev_status)
    for name, t, shape in (("q", q, (T, H, dk)), ("k", k, (T, H, dk)), ("v", v, (T, H, dv))):
        _need(t, name, shape, q.dtype, dev)
    _need_prefill_rest(T, H, dk, dv, q.dtype, dev, g, beta, cu_seqlens, state_indices, state_pool, out,
                       checkpoints, ckpt_offsets, gate, norm_w, has_initial_state, dev_status)
    return dev


def _need_prefill_rest(T, H, dk, dv, dtype, dev, g, beta, cu_seqlens, state_indices, state_pool, out,
                       checkpoints, ckpt_offsets, gate, norm_w, has_initial_state, dev_status):
    """The prefill's checks of every tensor but q, k and v."""
    N = state_indices.shape[0]
    _one_device(dev, g=g, beta=beta, cu_seqlens=cu_seqlens, state_indices=state_indices,
                state_pool=state_pool, out=out, checkpoints=checkpoints, ckpt_offsets=ckpt_offsets,
                gate=gate, norm_w=norm_w, has_initial_state=has_initial_state, dev_status=dev_status)
    for name, t, shape in (("g", g, (T, H, dk)), ("beta", beta, (T, H)), ("out", out, (T, H, dv)),
                           ("gate", gate, (T, H, dv)), ("norm_w", norm_w, (dv,))):
        _need(t, name, shape, dtype, dev)
    _need(cu_seqlens, "cu_seqlens", (N + 1,), torch.int32, dev)
    _need(state_indices, "state_indices", (N,), torch.int32, dev)
    _need(has_initial_state, "has_initial_state", (N,), torch.int32, dev)
    _need(ckpt_offsets, "ckpt_offsets", (N + 1,), torch.int32, dev)
    _need(state_pool, "state_pool", (None, H, dk, dv), None, dev)
    _need(checkpoints, "checkpoints", (None, H, dk, dv), state_pool.dtype, dev)
    _need(dev_status, "dev_status", None, torch.int32, dev)


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return KDA_F32
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float16:
        return KDA_F16
    raise ValueError(f"unsupported dtype {t.dtype}")


def _stream(stream, dev) -> ctypes.c_void_p:
    """Raw handle of ``stream`` (default: the current stream of ``dev``, the
    device of the call's tensors); a given stream must belong to ``dev``."""
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    elif stream.device != dev:
        raise ValueError(f"stream is on {stream.device} but the call's tensors are on {dev}")
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status: int, where: str):
    if status != KDA_OK:
        raise KdaError(status, where)


def kda_status_string(status: int) -> str:
    return load().kda_status_string(int(status)).decode()


def kda_version() -> int:
    return load().kda_version()


def kda_testing_set_first_wait_tries(tries: int, kernels: int = 3) -> None:
    """Testing only (see ``include/kda.h``): polls of the first bounded wait
    of the prefill kernels selected by ``kernels`` (bit 0 intra-chunk, bit 1
    state) launched from now on; a negative value restores the default."""
    load().kda_testing_set_first_wait_tries(int(tries), int(kernels))


def kda_prefill_workspace_bytes(N: int, T: int, H: int, dk: int, dv: int, chunk: int) -> int:
    return int(load().kda_prefill_workspace_bytes(N, T, H, dk, dv, chunk))


PREFILL_PATHS = {0: "unsupported", 1: "cuda cores", 2: "tensor cores"}


def kda_prefill_path(dk: int, dv: int, chunk: int, in_dtype) -> str:
    """Which kernels kda_prefill_chunked runs for this shape (the library's
    own answer): 'tensor cores', 'cuda cores' or 'unsupported'."""
    code = load().kda_prefill_path(int(dk), int(dv), int(chunk), _dtype_of(in_dtype))
    return PREFILL_PATHS[int(code)]


def _dtype_of(dt) -> int:
    return {torch.float32: KDA_F32, torch.bfloat16: KDA_BF16, torch.float16: KDA_F16}[dt]


def prefill_launches(dk: int, dv: int, chunk: int, in_dtype, gate: bool) -> int:
    """Kernel launches one kda_prefill_chunked call makes: the tensor-core path
    runs an intra-chunk and a state kernel; the CUDA-core path runs one kernel,
    plus a norm-gate pass when gated with dv = 128 (at dv <= 64 the kernel
    fuses the norm-gate)."""
    if kda_prefill_path(dk, dv, chunk, in_dtype) == "tensor cores":
        return 2
    return 2 if gate and dv > 64 else 1


def kda_prefill_chunked(q, k, v, g, beta, cu_seqlens, state_indices, state_pool, out, *,
                        chunk: int = 64, checkpoints=None, checkpoint_every: int = 0,
                        ckpt_offsets=None, gate=None, norm_w=None, eps: float = 1e-6,
                        gate_act: str = "sigmoid", has_initial_state=None, scale: float = 0.0,
                        workspace=None, dev_status=None, stream=None):
    """Chunked varlen prefill (see ``include/kda.h``).  All tensors on one
    CUDA device; ``state_pool`` is updated in place, ``out`` (and
    ``checkpoints``/``ckpt_offsets`` when given) are written."""
    dev = _need_prefill(q, k, v, g, beta, cu_seqlens, state_indices, state_pool, out, checkpoints,
                        ckpt_offsets, gate, norm_w, has_initial_state, dev_status)
    _need(workspace, "workspace", None, None, dev)
    T, H, dk = q.shape
    dv = v.shape[-1]
    N = state_indices.shape[0]
    cap = checkpoints.shape[0] if checkpoints is not None else 0
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    with torch.cuda.device(dev):
        st = load().kda_prefill_chunked(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _dtype(q), _ptr(cu_seqlens), N, T,
            _ptr(state_indices), _ptr(has_initial_state), _ptr(state_pool), state_pool.shape[0],
            _dtype(state_pool), _ptr(out), _ptr(checkpoints), int(checkpoint_every), cap,
            _ptr(ckpt_offsets), _ptr(gate), _ptr(norm_w), float(eps), GATE_ACT[gate_act], H, dk, dv,
            int(chunk), float(scale), _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream, dev))
    _check(st, "kda_prefill_chunked")


def kda_prefill_chunked_conv(x, conv_w, conv_state_pool, g, beta, cu_seqlens, state_indices, state_pool,
                             out, *, conv_b=None, conv_act: str = "silu", chunk: int = 64,
                             checkpoints=None, checkpoint_every: int = 0, ckpt_offsets=None, gate=None,
                             norm_w=None, eps: float = 1e-6, gate_act: str = "sigmoid",
                             has_initial_state=None, scale: float = 0.0, workspace=None,
                             dev_status=None, stream=None):
    """Short convolution, L2 normalisation of q and k, and the chunked prefill
    in one pass (see ``include/kda.h``).  ``x`` is the packed projection
    output [T, 3*H*d] (channels q, then k, then v); conv_w [3*H*d, W];
    conv_state_pool [slots, W-1, 3*H*d] is updated in place like state_pool.
    The shapes H, d come from ``g`` [T, H, d]."""
    T, H, dk = g.shape
    dev = g.device
    C3 = 3 * H * dk
    Wd = conv_w.shape[-1] if conv_w.dim() == 2 else 0
    _one_device(dev, x=x, conv_w=conv_w, conv_b=conv_b, conv_state_pool=conv_state_pool, beta=beta,
                cu_seqlens=cu_seqlens, state_indices=state_indices, state_pool=state_pool, out=out,
                checkpoints=checkpoints, ckpt_offsets=ckpt_offsets, gate=gate, norm_w=norm_w,
                has_initial_state=has_initial_state, dev_status=dev_status, workspace=workspace)
    for name, t, shape in (("x", x, (T, C3)), ("conv_w", conv_w, (C3, Wd)), ("conv_b", conv_b, (C3,)),
                           ("conv_state_pool", conv_state_pool, (None, Wd - 1, C3))):
        _need(t, name, shape, g.dtype, dev)
    _need_prefill_rest(T, H, dk, dk, g.dtype, dev, g, beta, cu_seqlens, state_indices, state_pool, out,
                       checkpoints, ckpt_offsets, gate, norm_w, has_initial_state, dev_status)
    _need(workspace, "workspace", None, None, dev)
    N = state_indices.shape[0]
    cap = checkpoints.shape[0] if checkpoints is not None else 0
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    if not x.is_contiguous():
        raise ValueError("libkda takes contiguous tensors")
    base = x.data_ptr() if x.numel() > 0 else None
    part = H * dk * x.element_size()
    xq, xk, xv = ((None, None, None) if base is None else
                  (ctypes.c_void_p(base), ctypes.c_void_p(base + part), ctypes.c_void_p(base + 2 * part)))
    with torch.cuda.device(dev):
        st = load().kda_prefill_chunked_conv(
            xq, xk, xv, C3, _ptr(conv_w), _ptr(conv_b), Wd, CONV_ACT[conv_act], _ptr(conv_state_pool),
            conv_state_pool.shape[0], _ptr(g), _ptr(beta), _dtype(g), _ptr(cu_seqlens), N, T,
            _ptr(state_indices), _ptr(has_initial_state), _ptr(state_pool), state_pool.shape[0],
            _dtype(state_pool), _ptr(out), _ptr(checkpoints), int(checkpoint_every), cap,
            _ptr(ckpt_offsets), _ptr(gate), _ptr(norm_w), float(eps), GATE_ACT[gate_act], H, dk, dk,
            int(chunk), float(scale), _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream, dev))
    _check(st, "kda_prefill_chunked_conv")


def kda_prefill_chunked_static_scratch(q, k, v, g, beta, cu_seqlens, state_indices, state_pool,
                                       out, *, chunk: int = 64, checkpoints=None,
                                       checkpoint_every: int = 0, ckpt_offsets=None, gate=None,
                                       norm_w=None, eps: float = 1e-6, gate_act: str = "sigmoid",
                                       has_initial_state=None, scale: float = 0.0,
                                       dev_status=None, stream=None):
    """kda_prefill_chunked for callers that cannot allocate: the library's own
    device array (STATIC_SCRATCH_BYTES) replaces the workspace.  Calls share
    that array, so calls that overlap on the GPU race; see include/kda.h."""
    dev = _need_prefill(q, k, v, g, beta, cu_seqlens, state_indices, state_pool, out, checkpoints,
                        ckpt_offsets, gate, norm_w, has_initial_state, dev_status)
    T, H, dk = q.shape
    dv = v.shape[-1]
    N = state_indices.shape[0]
    cap = checkpoints.shape[0] if checkpoints is not None else 0
    with torch.cuda.device(dev):
        st = load().kda_prefill_chunked_static_scratch(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _dtype(q), _ptr(cu_seqlens), N, T,
            _ptr(state_indices), _ptr(has_initial_state), _ptr(state_pool), state_pool.shape[0],
            _dtype(state_pool), _ptr(out), _ptr(checkpoints), int(checkpoint_every), cap,
            _ptr(ckpt_offsets), _ptr(gate), _ptr(norm_w), float(eps), GATE_ACT[gate_act], H, dk, dv,
            int(chunk), float(scale), _ptr(dev_status), _stream(stream, dev))
    _check(st, "kda_prefill_chunked_static_scratch")


def kda_decode_step(q, k, v, g, beta, state_indices, state_pool, out, *, gate=None, norm_w=None,
                    eps: float = 1e-6, gate_act: str = "sigmoid", scale: float = 0.0,
                    dev_status=None, stream=None):
    """One recurrent decode step for N one-token sequences (see ``include/kda.h``)."""
    N, H, dk = q.shape
    dv = v.shape[-1]
    dev = q.device
    _one_device(dev, k=k, v=v, g=g, beta=beta, state_indices=state_indices, state_pool=state_pool,
                out=out, gate=gate, norm_w=norm_w, dev_status=dev_status)
    for name, t, shape in (("q", q, (N, H, dk)), ("k", k, (N, H, dk)), ("g", g, (N, H, dk)),
                           ("v", v, (N, H, dv)), ("beta", beta, (N, H)), ("out", out, (N, H, dv)),
                           ("gate", gate, (N, H, dv)), ("norm_w", norm_w, (dv,))):
        _need(t, name, shape, q.dtype, dev)
    _need(state_indices, "state_indices", (N,), torch.int32, dev)
    _need(state_pool, "state_pool", (None, H, dk, dv), None, dev)
    _need(dev_status, "dev_status", None, torch.int32, dev)
    with torch.cuda.device(dev):
        st = load().kda_decode_step(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _dtype(q), _ptr(state_indices), N,
            _ptr(state_pool), state_pool.shape[0], _dtype(state_pool), _ptr(out), _ptr(gate),
            _ptr(norm_w), float(eps), GATE_ACT[gate_act], H, dk, dv, float(scale), _ptr(dev_status),
            _stream(stream, dev))
    _check(st, "kda_decode_step")


def kda_decode_multi(q, k, v, g, beta, state_indices, state_pool, out, token_states=None, *,
                     write_back: bool = False, gate=None, norm_w=None, eps: float = 1e-6,
                     gate_act: str = "sigmoid", scale: float = 0.0, dev_status=None, stream=None):
    """K decode steps per sequence with per-token states (see ``include/kda.h``).

    q, k, g are [N, K, H, dk]; v, out, gate [N, K, H, dv]; beta [N, K, H];
    token_states [N, K, H, dk, dv] or None.
    """
    N, K, H, dk = q.shape
    dv = v.shape[-1]
    dev = q.device
    _one_device(dev, k=k, v=v, g=g, beta=beta, state_indices=state_indices, state_pool=state_pool,
                out=out, token_states=token_states, gate=gate, norm_w=norm_w,
                dev_status=dev_status)
    for name, t, shape in (("q", q, (N, K, H, dk)), ("k", k, (N, K, H, dk)),
                           ("g", g, (N, K, H, dk)), ("v", v, (N, K, H, dv)),
                           ("beta", beta, (N, K, H)), ("out", out, (N, K, H, dv)),
                           ("gate", gate, (N, K, H, dv)), ("norm_w", norm_w, (dv,))):
        _need(t, name, shape, q.dtype, dev)
    _need(state_indices, "state_indices", (N,), torch.int32, dev)
    _need(state_pool, "state_pool", (None, H, dk, dv), None, dev)
    _need(token_states, "token_states", (N, K, H, dk, dv), state_pool.dtype, dev)
    _need(dev_status, "dev_status", None, torch.int32, dev)
    with torch.cuda.device(dev):
        st = load().kda_decode_multi(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _dtype(q), _ptr(state_indices), N, K,
            _ptr(state_pool), state_pool.shape[0], _dtype(state_pool), _ptr(out), _ptr(token_states),
            int(bool(write_back)), _ptr(gate), _ptr(norm_w), float(eps), GATE_ACT[gate_act], H, dk,
            dv, float(scale), _ptr(dev_status), _stream(stream, dev))
    _check(st, "kda_decode_multi")


def kda_commit_accepted(token_states, num_accepted, state_indices, state_pool, *,
                        dev_status=None, stream=None):
    """state_pool[idx_i] = token_states[i, a_i - 1] where a_i >= 1 (see ``include/kda.h``)."""
    N, K, H, dk, dv = token_states.shape
    dev = token_states.device
    _one_device(dev, num_accepted=num_accepted, state_indices=state_indices,
                state_pool=state_pool, dev_status=dev_status)
    _need(token_states, "token_states", None, None, dev)
    _need(num_accepted, "num_accepted", (N,), torch.int32, dev)
    _need(state_indices, "state_indices", (N,), torch.int32, dev)
    _need(state_pool, "state_pool", (None, H, dk, dv), token_states.dtype, dev)
    _need(dev_status, "dev_status", None, torch.int32, dev)
    with torch.cuda.device(dev):
        st = load().kda_commit_accepted(
            _ptr(token_states), _ptr(num_accepted), _ptr(state_indices), N, K, _ptr(state_pool),
            state_pool.shape[0], _dtype(state_pool), H, dk, dv, _ptr(dev_status), _stream(stream, dev))
    _check(st, "kda_commit_accepted")


CONV_ACT = {"none": 0, "silu": 1}


def kda_causal_conv1d_prefill(x, weight, cu_seqlens, state_indices, conv_state_pool, y, *, bias=None,
                              has_initial_state=None, act: str = "silu", dev_status=None,
                              stream=None):
    """Short causal convolution over packed sequences (see ``include/kda.h``):
    x, y [T, C]; weight [C, W]; conv_state_pool [slots, W-1, C]."""
    T, C = x.shape
    N = state_indices.shape[0]
    Wd = weight.shape[-1]
    dev = x.device
    _one_device(dev, weight=weight, cu_seqlens=cu_seqlens, state_indices=state_indices,
                conv_state_pool=conv_state_pool, y=y, bias=bias,
                has_initial_state=has_initial_state, dev_status=dev_status)
    for name, t, shape in (("x", x, (T, C)), ("y", y, (T, C)), ("weight", weight, (C, Wd)),
                           ("bias", bias, (C,)), ("conv_state_pool", conv_state_pool, (None, Wd - 1, C))):
        _need(t, name, shape, x.dtype, dev)
    _need(cu_seqlens, "cu_seqlens", (N + 1,), torch.int32, dev)
    _need(state_indices, "state_indices", (N,), torch.int32, dev)
    _need(has_initial_state, "has_initial_state", (N,), torch.int32, dev)
    _need(dev_status, "dev_status", None, torch.int32, dev)
    with torch.cuda.device(dev):
        st = load().kda_causal_conv1d_prefill(
            _ptr(x), _ptr(weight), _ptr(bias), _dtype(x), _ptr(cu_seqlens), N, T, C, weight.shape[1],
            _ptr(state_indices), _ptr(has_initial_state), _ptr(conv_state_pool), conv_state_pool.shape[0],
            CONV_ACT[act], _ptr(y), _ptr(dev_status), _stream(stream, dev))
    _check(st, "kda_causal_conv1d_prefill")


def kda_causal_conv1d_decode(x, weight, state_indices, conv_state_pool, y, *, bias=None,
                             act: str = "silu", dev_status=None, stream=None):
    """One token per sequence through the causal convolution: x, y [N, C]."""
    N, C = x.shape
    Wd = weight.shape[-1]
    dev = x.device
    _one_device(dev, weight=weight, state_indices=state_indices, conv_state_pool=conv_state_pool,
                y=y, bias=bias, dev_status=dev_status)
    for name, t, shape in (("x", x, (N, C)), ("y", y, (N, C)), ("weight", weight, (C, Wd)),
                           ("bias", bias, (C,)), ("conv_state_pool", conv_state_pool, (None, Wd - 1, C))):
        _need(t, name, shape, x.dtype, dev)
    _need(state_indices, "state_indices", (N,), torch.int32, dev)
    _need(dev_status, "dev_status", None, torch.int32, dev)
    with torch.cuda.device(dev):
        st = load().kda_causal_conv1d_decode(
            _ptr(x), _ptr(weight), _ptr(bias), _dtype(x), N, C, weight.shape[1], _ptr(state_indices),
            _ptr(conv_state_pool), conv_state_pool.shape[0], CONV_ACT[act], _ptr(y), _ptr(dev_status),
            _stream(stream, dev))
    _check(st, "kda_causal_conv1d_decode")


def kda_norm_gate_ex(o, gate, y, *, residual=None, residual_out=None, w=None, b=None,
                     eps: float = 1e-6, gate_act: str = "sigmoid", stream=None):
    """Norm-gate variants (see ``include/kda.h``): o, residual, residual_out, y
    are contiguous [rows, H, dv]; ``gate`` is a [rows, H, dv] tensor whose heads
    and values are contiguous and whose token rows may be further apart (a
    slice of a packed projection output): its row stride is passed as
    gate_row_stride."""
    rows, H, dv = o.shape
    dev = o.device
    _one_device(dev, gate=gate, y=y, residual=residual, residual_out=residual_out, w=w, b=b)
    for name, t, shape in (("o", o, (rows, H, dv)), ("y", y, (rows, H, dv)),
                           ("residual", residual, (rows, H, dv)),
                           ("residual_out", residual_out, (rows, H, dv)), ("w", w, (dv,)),
                           ("b", b, (dv,))):
        _need(t, name, shape, o.dtype, dev)
    _need(gate, "gate", (rows, H, dv), o.dtype, dev)
    if gate.stride(2) != 1 or gate.stride(1) != dv:
        raise ValueError("gate must be [rows, H, dv] with contiguous heads and values")
    gptr = ctypes.c_void_p(gate.data_ptr()) if gate.numel() > 0 else None
    with torch.cuda.device(dev):
        st = load().kda_norm_gate_ex(_ptr(o), _ptr(residual), _ptr(residual_out), gptr,
                                     int(gate.stride(0)) if rows > 1 else 0, _ptr(w), _ptr(b),
                                     float(eps), GATE_ACT[gate_act], _ptr(y), rows, H, dv, _dtype(o),
                                     _stream(stream, dev))
    _check(st, "kda_norm_gate_ex")


def kda_norm_gate(o, gate, w, y, *, eps: float = 1e-6, gate_act: str = "sigmoid", stream=None):
    """y = o / sqrt(mean(o^2)+eps) * w * act(gate) over the last dim of [rows, H, dv]."""
    rows, H, dv = o.shape
    dev = o.device
    _one_device(dev, gate=gate, w=w, y=y)
    for name, t, shape in (("o", o, (rows, H, dv)), ("gate", gate, (rows, H, dv)), ("w", w, (dv,)),
                           ("y", y, (rows, H, dv))):
        _need(t, name, shape, o.dtype, dev)
    with torch.cuda.device(dev):
        st = load().kda_norm_gate(_ptr(o), _ptr(gate), _ptr(w), float(eps), GATE_ACT[gate_act],
                                  _ptr(y), rows, H, dv, _dtype(o), _stream(stream, dev))
    _check(st, "kda_norm_gate")
