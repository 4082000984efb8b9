"""The C ABI on the host: libkda.so loads, exports every function that
include/kda.h declares, and rejects bad arguments with the documented status
before launching anything.  No GPU needed (no call here reaches a launch)."""
import ctypes
import os
import re

import pytest
import torch

import linear_attention_prefill_kda_gb300 as kda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 1 << 20  # an aligned, never-dereferenced stand-in for a device pointer
MIS = FAKE + 4  # misaligned


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(kda.lib_path()):
        from linear_attention_prefill_kda_gb300 import build
        build.build()
    return kda.load()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert {"kda_prefill_chunked", "kda_decode_step", "kda_norm_gate",
            "kda_prefill_workspace_bytes", "kda_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    assert kda.kda_status_string(0) == "ok"
    assert "unsupported" in kda.kda_status_string(-2)
    assert kda.kda_version() >= 100


def _prefill(lib, **over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, in_dtype=1, cu=FAKE, N=2, T=100, idx=FAKE,
             his=None, pool=FAKE, slots=4, sdt=0, out=FAKE, ck=None, every=0, cap=0, offs=None,
             gate=None, w=None, eps=1e-6, act=0, H=2, dk=64, dv=64, chunk=64, scale=0.0, ws=None,
             wsb=0, st=None)
    a.update(over)
    return lib.kda_prefill_chunked(
        a["q"], a["k"], a["v"], a["g"], a["beta"], a["in_dtype"], a["cu"], a["N"], a["T"],
        a["idx"], a["his"], a["pool"], a["slots"], a["sdt"], a["out"], a["ck"], a["every"],
        a["cap"], a["offs"], a["gate"], a["w"], a["eps"], a["act"], a["H"], a["dk"], a["dv"],
        a["chunk"], a["scale"], a["ws"], a["wsb"], a["st"], None)


@pytest.mark.parametrize("over,expect", [
    (dict(dk=32, dv=32), -2), (dict(dv=128), -2), (dict(chunk=32), -2), (dict(in_dtype=5), -2),
    (dict(sdt=7), -2), (dict(N=-1), -1), (dict(T=-5), -1), (dict(H=0), -1), (dict(slots=0), -1),
    (dict(q=None), -1), (dict(pool=None), -1), (dict(cu=None), -1), (dict(k=MIS), -1),
    (dict(out=MIS), -1), (dict(every=32), -1), (dict(every=128, ck=None, cap=10), -1),
    (dict(every=64, ck=FAKE, cap=0), -1), (dict(gate=FAKE), -1), (dict(w=FAKE), -1),
    (dict(gate=FAKE, w=FAKE, eps=-1.0), -1), (dict(st=MIS), -1), (dict(his=MIS), -1),
    (dict(act=2), -1), (dict(H=70000), -1),
])
def test_prefill_rejects(lib, over, expect):
    assert _prefill(lib, **over) == expect


def _decode(lib, **over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, in_dtype=1, idx=FAKE, N=4, pool=FAKE,
             slots=8, sdt=0, out=FAKE, gate=None, w=None, eps=1e-6, act=0, H=2, dk=128, dv=128,
             scale=0.0, st=None)
    a.update(over)
    return lib.kda_decode_step(a["q"], a["k"], a["v"], a["g"], a["beta"], a["in_dtype"], a["idx"],
                               a["N"], a["pool"], a["slots"], a["sdt"], a["out"], a["gate"],
                               a["w"], a["eps"], a["act"], a["H"], a["dk"], a["dv"], a["scale"],
                               a["st"], None)


@pytest.mark.parametrize("over,expect", [
    (dict(dk=64), -2), (dict(dk=96, dv=96), -2), (dict(in_dtype=3), -2), (dict(N=-2), -1),
    (dict(H=-1), -1), (dict(slots=0), -1), (dict(idx=None), -1), (dict(v=MIS), -1),
    (dict(gate=FAKE), -1), (dict(w=FAKE), -1), (dict(act=-1), -1),
])
def test_decode_rejects(lib, over, expect):
    assert _decode(lib, **over) == expect


def _decode_multi(lib, **over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, in_dtype=1, idx=FAKE, N=4, K=3, pool=FAKE,
             slots=8, sdt=0, out=FAKE, ts=FAKE, wb=0, gate=None, w=None, eps=1e-6, act=0, H=2,
             dk=128, dv=128, scale=0.0, st=None)
    a.update(over)
    return lib.kda_decode_multi(a["q"], a["k"], a["v"], a["g"], a["beta"], a["in_dtype"],
                                a["idx"], a["N"], a["K"], a["pool"], a["slots"], a["sdt"],
                                a["out"], a["ts"], a["wb"], a["gate"], a["w"], a["eps"], a["act"],
                                a["H"], a["dk"], a["dv"], a["scale"], a["st"], None)


@pytest.mark.parametrize("over,expect", [
    (dict(dk=64), -2), (dict(in_dtype=3), -2), (dict(sdt=4), -2), (dict(N=-1), -1),
    (dict(K=-1), -1), (dict(H=0), -1), (dict(slots=0), -1), (dict(idx=None), -1),
    (dict(ts=MIS), -1), (dict(q=MIS), -1), (dict(gate=FAKE), -1), (dict(act=3), -1),
    (dict(N=1 << 20, K=1 << 12), -1),
])
def test_decode_multi_rejects(lib, over, expect):
    assert _decode_multi(lib, **over) == expect


def _commit(lib, **over):
    a = dict(ts=FAKE, acc=FAKE, idx=FAKE, N=4, K=3, pool=FAKE, slots=8, sdt=0, H=2, dk=64, dv=64,
             st=None)
    a.update(over)
    return lib.kda_commit_accepted(a["ts"], a["acc"], a["idx"], a["N"], a["K"], a["pool"],
                                   a["slots"], a["sdt"], a["H"], a["dk"], a["dv"], a["st"], None)


@pytest.mark.parametrize("over,expect", [
    (dict(dv=128), -2), (dict(sdt=2), -2), (dict(N=-1), -1), (dict(slots=0), -1),
    (dict(ts=None), -1), (dict(acc=None), -1), (dict(pool=MIS), -1), (dict(st=MIS), -1),
])
def test_commit_rejects(lib, over, expect):
    assert _commit(lib, **over) == expect


def test_empty_calls_are_noops(lib):
    assert _decode(lib, N=0, q=None, k=None, v=None, g=None, beta=None, idx=None, out=None) == 0
    assert lib.kda_norm_gate(FAKE, FAKE, FAKE, 1e-6, 0, FAKE, 0, 4, 128, 1, None) == 0
    assert _decode_multi(lib, K=0, q=None, ts=None) == 0
    assert _decode_multi(lib, N=0, idx=None, out=None) == 0
    assert _commit(lib, N=0, ts=None, acc=None) == 0


@pytest.mark.parametrize("args,expect", [
    ((FAKE, FAKE, FAKE, 1e-6, 0, FAKE, 10, 4, 48, 1), -2),
    ((FAKE, FAKE, FAKE, 1e-6, 0, FAKE, 10, 4, 128, 9), -2),
    ((None, FAKE, FAKE, 1e-6, 0, FAKE, 10, 4, 128, 1), -1),
    ((FAKE, FAKE, MIS, 1e-6, 0, FAKE, 10, 4, 128, 1), -1),
    ((FAKE, FAKE, FAKE, -1.0, 0, FAKE, 10, 4, 128, 1), -1),
    ((FAKE, FAKE, FAKE, 1e-6, 0, FAKE, -1, 4, 128, 1), -1),
    ((FAKE, FAKE, FAKE, 1e-6, 5, FAKE, 10, 4, 128, 1), -1),
])
def test_norm_gate_rejects(lib, args, expect):
    assert lib.kda_norm_gate(*args, None) == expect


def _ngx(lib, **over):
    a = dict(o=FAKE, res=None, rout=None, gate=FAKE, gstride=0, w=None, b=None, eps=1e-6, act=0,
             y=FAKE, rows=10, H=4, dv=128, dt=2)
    a.update(over)
    return lib.kda_norm_gate_ex(a["o"], a["res"], a["rout"], a["gate"], a["gstride"], a["w"], a["b"],
                                a["eps"], a["act"], a["y"], a["rows"], a["H"], a["dv"], a["dt"], None)


@pytest.mark.parametrize("over,expect", [
    (dict(dv=48), -2), (dict(dt=3), -2), (dict(rows=-1), -1), (dict(H=0), -1), (dict(act=2), -1),
    (dict(eps=-1.0), -1), (dict(gstride=4 * 128 - 4), -1), (dict(gstride=4 * 128 + 2), -1),
    (dict(o=None), -1), (dict(gate=None), -1), (dict(y=MIS), -1), (dict(res=MIS), -1),
    (dict(rout=FAKE, y=FAKE), -1),
])
def test_norm_gate_ex_rejects(lib, over, expect):
    assert _ngx(lib, **over) == expect


def test_norm_gate_ex_empty_is_noop(lib):
    assert _ngx(lib, rows=0, o=None, gate=None, y=None) == 0


def _convp(lib, **over):
    a = dict(x=FAKE, w=FAKE, b=None, dt=1, cu=FAKE, N=3, T=100, C=256, W=4, idx=FAKE, his=None,
             pool=FAKE, slots=8, act=1, y=FAKE, st=None)
    a.update(over)
    return lib.kda_causal_conv1d_prefill(a["x"], a["w"], a["b"], a["dt"], a["cu"], a["N"], a["T"],
                                         a["C"], a["W"], a["idx"], a["his"], a["pool"], a["slots"],
                                         a["act"], a["y"], a["st"], None)


@pytest.mark.parametrize("over,expect", [
    (dict(W=5), -2), (dict(W=1), -2), (dict(C=100), -2), (dict(dt=2), -2), (dict(N=-1), -1),
    (dict(T=-1), -1), (dict(slots=0), -1), (dict(act=2), -1), (dict(w=None), -1),
    (dict(pool=None), -1), (dict(cu=None), -1), (dict(x=MIS), -1), (dict(b=MIS), -1),
    (dict(T=65536 * 64), -1),
])
def test_conv_prefill_rejects(lib, over, expect):
    assert _convp(lib, **over) == expect


@pytest.mark.parametrize("over,expect", [
    (dict(W=5), -2), (dict(C=12), -2), (dict(N=70000), -1), (dict(idx=None), -1), (dict(y=MIS), -1),
])
def test_conv_decode_rejects(lib, over, expect):
    a = dict(x=FAKE, w=FAKE, b=None, dt=0, N=3, C=256, W=4, idx=FAKE, pool=FAKE, slots=8, act=0,
             y=FAKE, st=None)
    a.update(over)
    assert lib.kda_causal_conv1d_decode(a["x"], a["w"], a["b"], a["dt"], a["N"], a["C"], a["W"],
                                        a["idx"], a["pool"], a["slots"], a["act"], a["y"], a["st"],
                                        None) == expect


def test_conv_empty_is_noop(lib):
    assert _convp(lib, T=0, x=None, y=None) == 0


def test_workspace_query(lib):
    assert kda.kda_prefill_workspace_bytes(8, 4096, 32, 128, 128, 64) >= 0
    assert lib.kda_prefill_workspace_bytes(-1, 10, 2, 64, 64, 64) == 0


def test_binding_refuses_missing_library(monkeypatch, tmp_path):
    """No silent fallback: without libkda.so every call raises."""
    monkeypatch.setattr(kda, "_lib", None)
    monkeypatch.setattr(kda, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        kda.kda_version()


def test_static_scratch_entry_rejects_oversize_on_host(lib):
    """The no-allocation prefill refuses a problem whose scratch exceeds its
    fixed array before touching the device."""
    rc = lib.kda_prefill_chunked_static_scratch(
        FAKE, FAKE, FAKE, FAKE, FAKE, 1, FAKE, 1, 65536, FAKE, None, FAKE, 4, 0, FAKE, None, 0, 0,
        None, None, None, 1e-6, 0, 32, 128, 128, 64, 0.0, None, None)
    assert rc == -3
    assert lib.kda_prefill_chunked_static_scratch(
        FAKE, FAKE, FAKE, FAKE, FAKE, 1, FAKE, 1, 100, FAKE, None, FAKE, 4, 0, FAKE, None, 0, 0,
        None, None, None, 1e-6, 0, 2, 96, 96, 64, 0.0, None, None) == -2


def test_prefill_conv_host_checks(lib):
    """The fused convolution + prefill refuses before touching the device: a
    width outside 2-4, a shape off the tensor-core path (d = 16, fp32 inputs)
    as unsupported; a row stride shorter than a head block or not a multiple
    of 8 elements, an unknown activation, a missing convolution pool or an
    empty one as invalid."""
    def call(width=4, act=1, stride=768, dk=128, in_dtype=1, cpool=FAKE, cslots=4):
        return lib.kda_prefill_chunked_conv(
            FAKE, FAKE, FAKE, stride, FAKE, None, width, act, cpool, cslots, FAKE, FAKE, in_dtype, FAKE, 1,
            64, FAKE, None, FAKE, 4, 0, FAKE, None, 0, 0, None, None, None, 1e-6, 0, 2, dk, dk, 64, 0.0,
            FAKE, 1 << 40, None, None)
    assert call(width=5) == -2 and call(width=1) == -2
    assert call(dk=16, stride=96) == -2 and call(in_dtype=0) == -2
    assert call(stride=100) == -1 and call(stride=260) == -1
    assert call(act=2) == -1 and call(cpool=None) == -1 and call(cslots=0) == -1


def test_binding_rejects_host_tensors_before_any_call():
    """The binding hands bare device pointers to the ABI: host tensors are
    refused with ValueError before the library is called."""
    import pytest as _pt
    q = torch.zeros(8, 2, 16, dtype=torch.bfloat16)
    b = torch.zeros(8, 2, dtype=torch.bfloat16)
    cu = torch.tensor([0, 8], dtype=torch.int32)
    idx = torch.zeros(1, dtype=torch.int32)
    pool = torch.zeros(2, 2, 16, 16)
    calls = [
        lambda: kda.kda_prefill_chunked(q, q, q, q, b, cu, idx, pool, q),
        lambda: kda.kda_prefill_chunked_static_scratch(q, q, q, q, b, cu, idx, pool, q),
        lambda: kda.kda_decode_step(q[:1], q[:1], q[:1], q[:1], b[:1], idx, pool, q[:1]),
        lambda: kda.kda_decode_multi(q[None, :1], q[None, :1], q[None, :1], q[None, :1], b[None, :1],
                                     idx, pool, q[None, :1]),
        lambda: kda.kda_commit_accepted(torch.zeros(1, 1, 2, 16, 16), idx, idx, pool),
        lambda: kda.kda_causal_conv1d_prefill(q[:, 0], q[0, :, :2].T.contiguous(), cu, idx,
                                              q[None, :1, 0], q[:, 0]),
        lambda: kda.kda_causal_conv1d_decode(q[:1, 0], q[0, :, :2].T.contiguous(), idx,
                                             q[None, :1, 0], q[:1, 0]),
        lambda: kda.kda_norm_gate(q, q, q[0, 0], q),
        lambda: kda.kda_norm_gate_ex(q, q, q),
        lambda: kda.kda_prefill_chunked_conv(torch.zeros(8, 96, dtype=torch.bfloat16),
                                             torch.zeros(96, 4, dtype=torch.bfloat16),
                                             torch.zeros(2, 3, 96, dtype=torch.bfloat16), q, b, cu, idx,
                                             pool, q),
    ]
    for call in calls:
        with _pt.raises(ValueError, match="CUDA tensor"):
            call()


def test_binding_rejects_tensors_on_two_devices():
    """Every tensor of a call must sit on the device of its first tensor: the
    ABI launches on one device and would read another device's pointers as its
    own.  The device check comes before the CUDA check, so a mix of host and
    'meta' tensors exercises it without a GPU; nothing reaches the library."""
    q = torch.zeros(8, 2, 16, dtype=torch.bfloat16)
    b = torch.zeros(8, 2, dtype=torch.bfloat16)
    cu = torch.tensor([0, 8], dtype=torch.int32)
    idx = torch.zeros(1, dtype=torch.int32)
    pool = torch.zeros(2, 2, 16, 16)
    qm = q.to("meta")
    calls = [
        lambda: kda.kda_prefill_chunked(q, qm, q, q, b, cu, idx, pool, q),
        lambda: kda.kda_prefill_chunked(q, q, q, q, b, cu, idx, pool.to("meta"), q),
        lambda: kda.kda_prefill_chunked(q, q, q, q, b, cu.to("meta"), idx, pool, q),
        lambda: kda.kda_prefill_chunked_static_scratch(q, q, q, q, b, cu, idx, pool, qm),
        lambda: kda.kda_decode_step(q[:1], q[:1], qm[:1], q[:1], b[:1], idx, pool, q[:1]),
        lambda: kda.kda_decode_multi(q[None, :1], q[None, :1], q[None, :1], q[None, :1],
                                     b[None, :1], idx.to("meta"), pool, q[None, :1]),
        lambda: kda.kda_commit_accepted(torch.zeros(1, 1, 2, 16, 16), idx, idx,
                                        pool.to("meta")),
        lambda: kda.kda_causal_conv1d_prefill(q[:, 0], q[0, :, :2].T.contiguous(), cu, idx,
                                              q[None, :1, 0], qm[:, 0]),
        lambda: kda.kda_causal_conv1d_decode(q[:1, 0], q[0, :, :2].T.contiguous(), idx,
                                             q[None, :1, 0].to("meta"), q[:1, 0]),
        lambda: kda.kda_norm_gate(q, qm, q[0, 0], q),
        lambda: kda.kda_norm_gate_ex(q, q, qm),
        lambda: kda.kda_prefill_chunked_conv(torch.zeros(8, 96, dtype=torch.bfloat16),
                                             torch.zeros(96, 4, dtype=torch.bfloat16),
                                             torch.zeros(2, 3, 96, dtype=torch.bfloat16), q, b, cu, idx,
                                             pool, qm),
    ]
    for call in calls:
        with pytest.raises(ValueError, match="one CUDA device"):
            call()


def test_prefill_path_query(lib):
    """The library's own answer to which kernels a prefill shape takes: the
    tensor-core kernels for bf16 inputs, dk = dv in {64, 128}, chunk 64; the
    CUDA-core kernel otherwise; unsupported shapes say so."""
    assert kda.kda_prefill_path(128, 128, 64, torch.bfloat16) == "tensor cores"
    assert kda.kda_prefill_path(64, 64, 64, torch.bfloat16) == "tensor cores"
    assert kda.kda_prefill_path(16, 16, 16, torch.float32) == "cuda cores"
    assert kda.kda_prefill_path(16, 16, 64, torch.bfloat16) == "cuda cores"
    assert kda.kda_prefill_path(128, 128, 16, torch.bfloat16) == "cuda cores"
    assert kda.kda_prefill_path(128, 128, 64, torch.float32) == "cuda cores"
    assert kda.kda_prefill_path(96, 96, 64, torch.bfloat16) == "unsupported"
    assert kda.kda_prefill_path(64, 128, 64, torch.bfloat16) == "unsupported"
    assert kda.prefill_launches(64, 64, 64, torch.bfloat16, gate=False) == 2
    # CUDA-core path: the norm-gate is fused up to dv = 64, a second pass at dv = 128
    assert kda.prefill_launches(16, 16, 16, torch.float32, gate=True) == 1
    assert kda.prefill_launches(64, 64, 16, torch.bfloat16, gate=True) == 1
    assert kda.prefill_launches(128, 128, 64, torch.float32, gate=True) == 2
    assert kda.prefill_launches(128, 128, 64, torch.float32, gate=False) == 1
