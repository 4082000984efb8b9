"""GPU parity: libkda through its C ABI against the fp64 oracle on the same
seeded inputs.  Values within the tolerance rule of kda_testutil; indexing,
checkpoint placement, padding rows and untouched pool slots bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from kda_testutil import (excess_error, max_abs, oracle_prefill, oracle_prefill_conv, record, run_prefill,
                          run_prefill_conv, to_dev, tol_for)

W_ = W  # the workloads module, for tests whose parameter W is a convolution width

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _check_prefill(kda, w, d, *, heads=None, ckpt=True, label=None):
    pool0 = d["pool"].clone()
    out, pool, ck, offs, status = run_prefill(kda, d, w, DEV, ckpt=ckpt)
    assert int(status.item()) == 0, kda.DEV_STATUS[int(status.item())]
    o_ref, p_ref, ck_ref, offs_ref = oracle_prefill(oracle, d, w, ckpt=ckpt, heads=heads)
    tol = tol_for(w.state_dtype)
    hsel = slice(None) if heads is None else heads
    idx = d["state_indices"].tolist()
    lens = (d["cu_seqlens"][1:] - d["cu_seqlens"][:-1]).tolist()
    # outputs
    if label:
        record(label, "out", out[:, hsel], o_ref)
    assert excess_error(out[:, hsel], o_ref) <= tol
    # touched slots, untouched slots bit-exact
    touched = [s for s, L in zip(idx, lens) if s >= 0 and L > 0]
    pool_cpu = pool.cpu()
    for s in range(w.num_slots):
        if s in touched:
            if label:
                record(label, "final_state", pool_cpu[s][hsel], p_ref[s])
            assert excess_error(pool_cpu[s][hsel], p_ref[s]) <= tol, s
        else:
            assert torch.equal(pool_cpu[s], pool0[s]), f"slot {s} modified"
    # checkpoints: offsets bit-exact, values within tolerance
    if ckpt and w.checkpoint_every:
        assert offs.cpu().numpy().tolist() == offs_ref.tolist()
        n = int(offs_ref[-1])
        if n:
            real = []
            for i, s in enumerate(idx):
                if s >= 0:
                    real.extend(range(int(offs_ref[i]), int(offs_ref[i + 1])))
            if label:
                record(label, "checkpoints", ck[real][:, hsel], ck_ref[real])
            assert excess_error(ck[real][:, hsel], ck_ref[real]) <= tol
    return out, pool


def test_prefill_tiny(kda_gpu):
    _check_prefill(kda_gpu, W.TINY, W.make_prefill(W.TINY), label=W.TINY.name)


def test_prefill_varlen(kda_gpu):
    # d = 64, bf16, chunk 64: the tensor-core kernels (tiles zero-padded to 128 channels)
    assert kda_gpu.kda_prefill_path(64, 64, 64, torch.bfloat16) == "tensor cores"
    _check_prefill(kda_gpu, W.VARLEN, W.make_prefill(W.VARLEN), label=W.VARLEN.name)


def test_prefill_d64_tensor_cores_gate_and_bf16_state(kda_gpu):
    """The d = 64 tensor-core path with the fused norm-gate (mean over 64
    columns), bf16 state and checkpoints, lengths around the chunk edges and a
    padding sequence."""
    w = W.SCHED.replace(seqlens=(1, 63, 64, 65, 0, 200, 130), H=6, dk=64, dv=64, num_slots=12,
                        slot_range=None, state_dtype=torch.bfloat16, checkpoint_every=64, seed=264)
    d = W.make_prefill(w)
    d["state_indices"][4] = -1
    _check_prefill(kda_gpu, w, d)


def test_prefill_sched_full(kda_gpu):
    _check_prefill(kda_gpu, W.SCHED, W.make_prefill(W.SCHED), label=W.SCHED.name)


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("chunk,d", [(64, 64), (64, 128), (16, 64), (16, 128), (64, 16), (16, 16)])
def test_prefill_edge_lengths(kda_gpu, chunk, d, state_dtype):
    """Empty segments, lengths 1, C-1, C, C+1, a padding sequence (-1) and the
    highest slot id, with checkpoints every 2C."""
    lens = (0, 1, chunk - 1, chunk, chunk + 1, 7, 3 * chunk + 5)
    w = W.VARLEN.replace(seqlens=lens, H=3, dk=d, dv=d, chunk=chunk, checkpoint_every=2 * chunk,
                         state_dtype=state_dtype, num_slots=12, seed=40 + d + chunk)
    d_ = W.make_prefill(w)
    idx = d_["state_indices"].clone()
    idx[5] = -1
    idx[6] = w.num_slots - 1
    idx[:5] = torch.tensor([0, 3, 5, 7, 9], dtype=torch.int32)
    d_["state_indices"] = idx
    out, _ = _check_prefill(kda_gpu, w, d_)
    t0, t1 = int(d_["cu_seqlens"][5]), int(d_["cu_seqlens"][6])
    assert torch.count_nonzero(out[t0:t1].float()).item() == 0  # padding rows exactly zero


def test_prefill_many_sequences(kda_gpu):
    """100 sequences of 1-150 tokens (the slot lookup scans 32 sequences per
    step), a few empty ones and padding rows, tensor-core shape, checkpoints
    every 128 tokens, SiLU gate and a mix of initial-state flags."""
    gen = torch.Generator().manual_seed(61)
    lens = torch.randint(1, 151, (100,), generator=gen)
    lens[[7, 50, 93]] = 0
    w = W.SCHED.replace(seqlens=tuple(int(x) for x in lens), H=2, num_slots=128, slot_range=None,
                        checkpoint_every=128, seed=62)
    d = W.make_prefill(w)
    idx = d["state_indices"].clone()
    idx[[3, 64]] = -1
    d["state_indices"] = idx
    d["gate_act"] = "silu"
    d["has_initial_state"] = (torch.arange(100) % 3 != 0).to(torch.int32)
    out, _ = _check_prefill(kda_gpu, w, d)
    for i in (3, 64):
        t0, t1 = int(d["cu_seqlens"][i]), int(d["cu_seqlens"][i + 1])
        assert torch.count_nonzero(out[t0:t1].float()).item() == 0


def test_prefill_tc_shape_mixed(kda_gpu):
    """The tensor-core shape (d=128, chunk 64, bf16) with short, partial and
    multi-chunk sequences, bf16 state, checkpoints and the fused norm-gate."""
    w = W.SCHED.replace(seqlens=(1, 63, 64, 65, 0, 200, 511), H=4, num_slots=16, slot_range=None,
                        state_dtype=torch.bfloat16, checkpoint_every=128, seed=123)
    _check_prefill(kda_gpu, w, W.make_prefill(w))


@pytest.mark.parametrize("d,in_dtype,state_dtype", [(128, torch.bfloat16, torch.float32),
                                                    (128, torch.bfloat16, torch.bfloat16),
                                                    (64, torch.bfloat16, torch.float32),
                                                    (16, torch.float32, torch.float32)])
def test_prefill_new_prompts_and_silu_gate(kda_gpu, d, in_dtype, state_dtype):
    """Sequences flagged without initial state start from zero whatever their
    slot holds (the slots hold random states here); the SiLU gate activation."""
    w = W.SCHED.replace(seqlens=(70, 1, 130, 33), H=3, dk=d, dv=d, in_dtype=in_dtype,
                        state_dtype=state_dtype, num_slots=9, slot_range=None,
                        checkpoint_every=64, seed=600 + d)
    dd = W.make_prefill(w)
    dd["has_initial_state"] = torch.tensor([0, 0, 1, 0], dtype=torch.int32)
    dd["gate_act"] = "silu"
    _check_prefill(kda_gpu, w, dd)


@pytest.mark.parametrize("d,chunk,in_dtype,act", [(16, 64, torch.bfloat16, "silu"),
                                                  (64, 16, torch.bfloat16, "sigmoid"),
                                                  (128, 64, torch.float32, "silu"),
                                                  (128, 16, torch.bfloat16, "sigmoid")])
def test_prefill_cuda_core_norm_gate(kda_gpu, d, chunk, in_dtype, act):
    """The CUDA-core prefill's output norm-gate: fused into the kernel where one
    64-column slab holds the whole row (dv <= 64, one launch), a second pass at
    dv = 128 (through fp32 scratch for bf16 inputs)."""
    assert kda_gpu.kda_prefill_path(d, d, chunk, in_dtype) == "cuda cores"
    assert kda_gpu.prefill_launches(d, d, chunk, in_dtype, True) == (1 if d <= 64 else 2)
    w = W.SCHED.replace(seqlens=(90, 17, 140), H=3, dk=d, dv=d, chunk=chunk, in_dtype=in_dtype,
                        checkpoint_every=2 * chunk, num_slots=6, slot_range=None, seed=700 + d + chunk)
    dd = W.make_prefill(w)
    dd["gate_act"] = act
    _check_prefill(kda_gpu, w, dd)


def test_prefill_gate_fp32_and_chunk16(kda_gpu):
    w = W.SCHED.replace(seqlens=(100, 37, 256), H=4, dk=64, dv=64, chunk=16, checkpoint_every=32,
                        in_dtype=torch.float32, num_slots=8, slot_range=None, seed=77)
    _check_prefill(kda_gpu, w, W.make_prefill(w))


@pytest.mark.parametrize("d,in_dtype", [(64, torch.float32), (128, torch.bfloat16)])
def test_prefill_extreme_decay(kda_gpu, d, in_dtype):
    """g = -1e30 on some tokens (alpha = 0 exactly) must erase history without
    producing inf/nan (the d=128 bf16 case exercises the exact fallback of the
    factorised decay in the tensor-core path)."""
    w = W.VARLEN.replace(seqlens=(130, 70), H=2, dk=d, dv=d, in_dtype=in_dtype, seed=91,
                         checkpoint_every=0)
    d = W.make_prefill(w)
    d["g"][10] = -1e30
    d["g"][64, :, :5] = -1e30
    d["g"][100:103] = -40.0
    out, _ = _check_prefill(kda_gpu, w, d, ckpt=False)
    assert torch.isfinite(out.float()).all()


def test_prefill_bad_index_latches_status(kda_gpu):
    w = W.VARLEN.replace(seqlens=(20, 30), H=2, seed=5, checkpoint_every=0)
    d = W.make_prefill(w)
    d["state_indices"] = torch.tensor([1, w.num_slots + 3], dtype=torch.int32)
    pool0 = d["pool"].clone()
    out, pool, _, _, status = run_prefill(kda_gpu, d, w, DEV, ckpt=False)
    assert int(status.item()) == 1
    assert torch.count_nonzero(out[20:].float()).item() == 0
    p = pool.cpu()
    for s in range(w.num_slots):
        if s != 1:
            assert torch.equal(p[s], pool0[s])


@pytest.mark.parametrize("d,in_dtype", [(128, torch.bfloat16), (64, torch.float32)],
                         ids=["tensor-cores", "cuda-cores"])
def test_duplicate_slot_latches_status(kda_gpu, d, in_dtype):
    """Two sequences of one call naming the same state slot (or conv cache
    slot) would race on it: every kernel family reports KDA_DEV_DUP_INDEX (5).
    The values of the sequences involved are undefined; the other slots stay
    untouched."""
    w = W.SCHED.replace(seqlens=(70, 30, 40), H=2, dk=d, dv=d, in_dtype=in_dtype, num_slots=8,
                        slot_range=None, checkpoint_every=0, seed=55)
    dd = W.make_prefill(w)
    dd["state_indices"] = torch.tensor([3, 5, 3], dtype=torch.int32)
    pool0 = dd["pool"].clone()
    out, pool, _, _, status = run_prefill(kda_gpu, dd, w, DEV, ckpt=False)
    assert int(status.item()) == 5
    p = pool.cpu()
    for slot in range(w.num_slots):
        if slot not in (3, 5):
            assert torch.equal(p[slot], pool0[slot])
    # decode, verification + commit, convolution: the same report
    dw = W.DECODE.replace(N=3, H=2, dk=64, dv=64, num_slots=8)
    pd = W.make_decode_pool(dw)
    idx = torch.tensor([6, 1, 6], dtype=torch.int32, device=DEV)
    for kind in ("decode", "verify", "commit"):
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        dpool = pd["pool"].to(DEV)
        if kind == "decode":
            sd = to_dev(W.make_decode_step(dw, 0), DEV)
            o = torch.empty(dw.N, dw.H, dw.dv, device=DEV, dtype=dw.in_dtype)
            kda_gpu.kda_decode_step(sd["q"], sd["k"], sd["v"], sd["g"], sd["beta"], idx, dpool, o,
                                    dev_status=status)
        else:
            dr = W.make_decode_draft(dw, 2)
            dr.pop("num_accepted")
            t = to_dev(dr, DEV)
            o = torch.empty(dw.N, 2, dw.H, dw.dv, device=DEV, dtype=dw.in_dtype)
            ts = torch.empty(dw.N, 2, dw.H, dw.dk, dw.dv, device=DEV, dtype=dw.state_dtype)
            if kind == "verify":
                kda_gpu.kda_decode_multi(t["q"], t["k"], t["v"], t["g"], t["beta"], idx, dpool, o, ts,
                                         dev_status=status)
            else:
                kda_gpu.kda_decode_multi(t["q"], t["k"], t["v"], t["g"], t["beta"],
                                         torch.tensor([6, 1, 2], dtype=torch.int32, device=DEV), dpool,
                                         o, ts)
                acc = torch.tensor([1, 0, 2], dtype=torch.int32, device=DEV)
                kda_gpu.kda_commit_accepted(ts, acc, idx, dpool, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 5, kind
    # a repeated slot whose second user commits nothing is not a conflict
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda_gpu.kda_commit_accepted(ts, torch.tensor([1, 0, 0], dtype=torch.int32, device=DEV), idx,
                                dpool, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    cd = W.make_conv((20, 9, 33), 64, 4, torch.bfloat16, num_slots=6, seed=3)
    cd = to_dev(cd, DEV)
    cidx = torch.tensor([2, 4, 2], dtype=torch.int32, device=DEV)
    for prefill in (True, False):
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        if prefill:
            y = torch.empty_like(cd["x"])
            kda_gpu.kda_causal_conv1d_prefill(cd["x"], cd["w"], cd["cu_seqlens"], cidx, cd["pool"], y,
                                              bias=cd["b"], dev_status=status)
        else:
            x1 = cd["x"][:3].contiguous()
            y1 = torch.empty_like(x1)
            kda_gpu.kda_causal_conv1d_decode(x1, cd["w"], cidx, cd["pool"], y1, bias=cd["b"],
                                             dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 5, ("conv", prefill)


def test_prefill_longprompt_bf16_state(kda_gpu):
    """One 32768-token sequence as 8 calls of 4096 carrying bf16 state through
    the pool, against the one-shot fp64 oracle (every head) and against a
    single 32768-token call; checkpoint positions bit-exact."""
    w = W.LONGPROMPT
    d = W.make_prefill(w)
    pool_init = d["pool"].clone()
    slot = int(d["state_indices"][0])
    T, seg = w.T, 4096
    dev_pool = pool_init.to(DEV)
    idx = d["state_indices"].to(DEV)
    outs, cks = [], []
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(kda_gpu.kda_prefill_workspace_bytes(1, seg, w.H, w.dk, w.dv, w.chunk),
                     dtype=torch.uint8, device=DEV)
    for c in range(T // seg):
        sl = slice(c * seg, (c + 1) * seg)
        t = {k: d[k][sl].to(DEV) for k in ("q", "k", "v", "g", "beta")}
        out = torch.empty(seg, w.H, w.dv, device=DEV, dtype=w.in_dtype)
        ck = torch.empty(seg // w.checkpoint_every, w.H, w.dk, w.dv, device=DEV, dtype=w.state_dtype)
        kda_gpu.kda_prefill_chunked(t["q"], t["k"], t["v"], t["g"], t["beta"],
                                    W.cu_from_lengths([seg]).to(DEV), idx, dev_pool, out,
                                    chunk=w.chunk, checkpoints=ck,
                                    checkpoint_every=w.checkpoint_every, workspace=ws,
                                    dev_status=status)
        outs.append(out)
        cks.append(ck)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    out8 = torch.cat(outs)
    ck8 = torch.cat(cks)
    # one-shot GPU call
    pool1 = pool_init.to(DEV)
    out1, pool1, ck1, offs1, st1 = run_prefill(kda_gpu, dict(d, pool=pool_init.clone()), w, DEV)
    assert int(st1.item()) == 0
    assert offs1.cpu().tolist() == [0, T // w.checkpoint_every]
    assert ck1.shape[0] == ck8.shape[0] == T // w.checkpoint_every
    tol = tol_for(w.state_dtype)
    # the two GPU runs agree
    assert max_abs(out8, out1.double().cpu().numpy()) <= tol
    assert max_abs(ck8, ck1.double().cpu().numpy()) <= tol
    # against the fp64 oracle, all 32 heads
    o_ref, p_ref, ck_ref, _ = oracle_prefill(oracle, d, w)
    for name, x, ref in (("out (8 calls)", out8, o_ref), ("out (one call)", out1, o_ref),
                         ("checkpoints (8 calls)", ck8, ck_ref), ("checkpoints (one call)", ck1, ck_ref),
                         ("final_state (8 calls)", dev_pool[slot], p_ref[slot]),
                         ("final_state (one call)", pool1[slot], p_ref[slot])):
        record(w.name, name, x, ref)
    assert excess_error(out8, o_ref) <= tol
    assert excess_error(out1, o_ref) <= tol
    assert excess_error(ck8, ck_ref) <= tol
    assert excess_error(ck1, ck_ref) <= tol
    assert excess_error(dev_pool[slot], p_ref[slot]) <= tol
    assert excess_error(pool1[slot], p_ref[slot]) <= tol


def test_decode_full_64_steps(kda_gpu):
    """256 sequences x 64 in-place steps on a 1024-slot fp32 pool; the oracle
    follows every sequence and head at every step."""
    w = W.DECODE
    pd = W.make_decode_pool(w)
    pool0 = pd["pool"]
    idx = pd["state_indices"]
    sample = list(range(w.N))
    ref_pool = pool0[idx[sample].long()].double().numpy().copy()
    ref_idx = np.arange(len(sample), dtype=np.int32)
    dev_pool = pool0.to(DEV)
    didx = idx.to(DEV)
    nw = pd["norm_w"].to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.empty(w.N, w.H, w.dv, device=DEV, dtype=w.in_dtype)
    tol = tol_for(w.state_dtype)
    worst = 0.0
    for step in range(w.steps):
        sd = W.make_decode_step(w, step)
        t = to_dev(sd, DEV)
        kda_gpu.kda_decode_step(t["q"], t["k"], t["v"], t["g"], t["beta"], didx, dev_pool, out,
                                gate=t["gate"], norm_w=nw, eps=pd["eps"], dev_status=status)
        y_ref, ref_pool = oracle.decode(*(sd[k][sample] for k in ("q", "k", "v", "g", "beta")),
                                        ref_idx, ref_pool, gate=sd["gate"][sample],
                                        norm_w=pd["norm_w"], eps=pd["eps"])
        worst = max(worst, excess_error(out[sample], y_ref))
        record(w.name, "out (every step)", out[sample], y_ref)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert worst <= tol, worst
    final = dev_pool[didx[sample].long()]
    record(w.name, "final_state", final, ref_pool)
    assert excess_error(final, ref_pool) <= tol
    # slots outside the batch are untouched, byte for byte
    mask = torch.ones(w.num_slots, dtype=torch.bool)
    mask[idx.long()] = False
    assert torch.equal(dev_pool[mask.to(DEV)].cpu(), pool0[mask])


@pytest.mark.parametrize("act", ["sigmoid", "silu"])
def test_decode_gate_activations(kda_gpu, act):
    w = W.DECODE.replace(N=6, H=2, num_slots=8, seed=710)
    pd = W.make_decode_pool(w)
    sd = W.make_decode_step(w, 0)
    pool = pd["pool"].to(DEV)
    t = to_dev(sd, DEV)
    out = torch.empty(w.N, w.H, w.dv, device=DEV, dtype=w.in_dtype)
    kda_gpu.kda_decode_step(t["q"], t["k"], t["v"], t["g"], t["beta"], pd["state_indices"].to(DEV),
                            pool, out, gate=t["gate"], norm_w=pd["norm_w"].to(DEV), eps=pd["eps"],
                            gate_act=act)
    torch.cuda.synchronize()
    y_ref, p_ref = oracle.decode(sd["q"], sd["k"], sd["v"], sd["g"], sd["beta"], pd["state_indices"],
                                 pd["pool"], gate=sd["gate"], norm_w=pd["norm_w"], eps=pd["eps"],
                                 gate_act=act)
    assert excess_error(out, y_ref) <= 0.01
    assert excess_error(pool, p_ref) <= 0.01


@pytest.mark.parametrize("d", [16, 64, 128])
@pytest.mark.parametrize("in_dtype,state_dtype", [(torch.float32, torch.float32),
                                                  (torch.bfloat16, torch.bfloat16),
                                                  (torch.float32, torch.bfloat16)])
def test_decode_small(kda_gpu, d, in_dtype, state_dtype):
    w = W.DECODE.replace(N=9, H=3, dk=d, dv=d, in_dtype=in_dtype, state_dtype=state_dtype,
                         num_slots=20, seed=300 + d)
    pd = W.make_decode_pool(w)
    sd = W.make_decode_step(w, 0)
    idx = torch.tensor([3, 0, 7, 12, -1, 19, 5, 8, 2], dtype=torch.int32)  # -1 pads, 19 = top slot
    pool = pd["pool"].to(DEV)
    t = to_dev(sd, DEV)
    out = torch.full((w.N, w.H, w.dv), float("nan"), device=DEV, dtype=in_dtype)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    for gated in (False, True):
        pool = pd["pool"].to(DEV)
        kda_gpu.kda_decode_step(t["q"], t["k"], t["v"], t["g"], t["beta"], idx.to(DEV), pool, out,
                                gate=t["gate"] if gated else None,
                                norm_w=pd["norm_w"].to(DEV) if gated else None, eps=pd["eps"],
                                dev_status=status)
        torch.cuda.synchronize()
        y_ref, p_ref = oracle.decode(sd["q"], sd["k"], sd["v"], sd["g"], sd["beta"], idx,
                                     pd["pool"], gate=sd["gate"] if gated else None,
                                     norm_w=pd["norm_w"] if gated else None, eps=pd["eps"])
        tol = tol_for(state_dtype)
        assert int(status.item()) == 0
        assert excess_error(out, y_ref) <= tol
        assert torch.count_nonzero(out[4].float()).item() == 0
        assert excess_error(pool, p_ref) <= tol


@pytest.mark.parametrize("d", [16, 64, 128])
@pytest.mark.parametrize("K", [1, 5])
@pytest.mark.parametrize("in_dtype,state_dtype", [(torch.float32, torch.float32),
                                                  (torch.bfloat16, torch.bfloat16),
                                                  (torch.bfloat16, torch.float32)])
def test_decode_multi_and_commit(kda_gpu, d, K, in_dtype, state_dtype):
    """K draft tokens per sequence: outputs and every per-token state against
    the oracle, the pool untouched by the verification call, then the commit
    of the accepted prefixes; a second call with write_back leaves the
    K-token state in the slots."""
    w = W.DECODE.replace(N=7, H=3, dk=d, dv=d, in_dtype=in_dtype,
                         state_dtype=state_dtype, num_slots=12, seed=900 + d + K)
    pd = W.make_decode_pool(w)
    dd = W.make_decode_draft(w, K)
    idx = torch.tensor([3, -1, 11, 0, 7, 5, 9], dtype=torch.int32)
    acc = dd["num_accepted"]
    t = to_dev(dd, DEV)
    nw = pd["norm_w"].to(DEV)
    pool = pd["pool"].to(DEV)
    out = torch.full((w.N, K, w.H, w.dv), float("nan"), device=DEV, dtype=in_dtype)
    ts = torch.full((w.N, K, w.H, w.dk, w.dv), float("nan"), device=DEV, dtype=state_dtype)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda_gpu.kda_decode_multi(t["q"], t["k"], t["v"], t["g"], t["beta"], idx.to(DEV), pool, out, ts,
                             gate=t["gate"], norm_w=nw, eps=pd["eps"], gate_act="silu",
                             dev_status=status)
    torch.cuda.synchronize()
    y_ref, ts_ref, pool_k = oracle.decode_multi(
        dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], idx, pd["pool"], gate=dd["gate"],
        norm_w=pd["norm_w"], eps=pd["eps"], gate_act="silu")
    tol = tol_for(state_dtype)
    live = (idx >= 0).numpy()
    assert int(status.item()) == 0
    assert excess_error(out, y_ref) <= tol
    assert torch.count_nonzero(out[1].float()).item() == 0
    assert excess_error(ts[torch.from_numpy(live).to(DEV)], ts_ref[live]) <= tol
    assert torch.isnan(ts[1].float()).all()  # padding rows keep no states
    assert torch.equal(pool.cpu(), pd["pool"])  # verification only reads the pool
    kda_gpu.kda_commit_accepted(ts, acc.to(DEV), idx.to(DEV), pool, dev_status=status)
    torch.cuda.synchronize()
    ref_commit = oracle.commit_accepted(ts_ref, acc.numpy(), idx.numpy(), pd["pool"])
    assert int(status.item()) == 0
    assert excess_error(pool, ref_commit) <= tol
    for i in range(w.N):  # slots with nothing accepted stay bit-identical
        if idx[i] >= 0 and acc[i] == 0:
            assert torch.equal(pool[idx[i]].cpu(), pd["pool"][idx[i]])
    pool2 = pd["pool"].to(DEV)
    kda_gpu.kda_decode_multi(t["q"], t["k"], t["v"], t["g"], t["beta"], idx.to(DEV), pool2, out,
                             None, write_back=True, gate=t["gate"], norm_w=nw, eps=pd["eps"],
                             gate_act="silu", dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert excess_error(pool2, pool_k) <= tol
    assert excess_error(out, y_ref) <= tol


def test_decode_multi_full_width(kda_gpu):
    """256 sequences x 4 draft tokens at 32 heads, d = 128 (the decode batch);
    every sequence against the oracle, in groups of 32 so that the fp64
    per-token states stay at half a gigabyte per group."""
    w, K = W.DECODE, 4
    pd = W.make_decode_pool(w)
    dd = W.make_decode_draft(w, K)
    idx = pd["state_indices"]
    t = to_dev(dd, DEV)
    pool = pd["pool"].to(DEV)
    out = torch.empty(w.N, K, w.H, w.dv, device=DEV, dtype=w.in_dtype)
    ts = torch.empty(w.N, K, w.H, w.dk, w.dv, device=DEV, dtype=w.state_dtype)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda_gpu.kda_decode_multi(t["q"], t["k"], t["v"], t["g"], t["beta"], idx.to(DEV), pool, out, ts,
                             gate=t["gate"], norm_w=pd["norm_w"].to(DEV), eps=pd["eps"],
                             dev_status=status)
    kda_gpu.kda_commit_accepted(ts, dd["num_accepted"].to(DEV), idx.to(DEV), pool,
                                dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    tol = tol_for(w.state_dtype)
    for g0 in range(0, w.N, 32):
        sample = list(range(g0, g0 + 32))
        sidx = idx[sample]
        sub_pool = pd["pool"][sidx.long()]
        ref_idx = np.arange(len(sample), dtype=np.int32)
        y_ref, ts_ref, _ = oracle.decode_multi(
            *(dd[n][sample] for n in ("q", "k", "v", "g", "beta")), ref_idx, sub_pool,
            gate=dd["gate"][sample], norm_w=pd["norm_w"], eps=pd["eps"])
        assert excess_error(out[sample], y_ref) <= tol
        assert excess_error(ts[sample], ts_ref) <= tol
        ref_commit = oracle.commit_accepted(ts_ref, dd["num_accepted"][sample].numpy(), ref_idx,
                                            sub_pool)
        assert excess_error(pool[sidx.long().to(DEV)], ref_commit) <= tol


@pytest.mark.parametrize("W", [2, 3, 4])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("act", ["none", "silu"])
def test_conv_prefill(kda_gpu, W, dtype, act):
    """Lengths 0, 1, W-2, W-1, 63, 64, 65, 200 (tiles of 64 tokens, inputs before
    a tile from x or the cache), one padding sequence, one without initial
    state; outputs and caches against the oracle, untouched slots unchanged.
    1032 channels leave a last block of 8; width 3 runs without bias."""
    lens = (0, 1, max(W - 2, 1), W - 1, 63, 64, 65, 200, 9)
    his = [1, 1, 0, 1, 1, 1, 0, 1, 1]
    d = W_.make_conv(lens, 1032, W, dtype, num_slots=16, seed=800 + W, has_initial=his)
    if W == 3:
        d["b"] = None
    idx = d["state_indices"].clone()
    idx[8] = -1
    d["state_indices"] = idx
    t = to_dev(d, DEV)
    y = torch.full_like(t["x"], float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda_gpu.kda_causal_conv1d_prefill(t["x"], t["w"], t["cu_seqlens"], t["state_indices"], t["pool"],
                                      y, bias=t["b"], has_initial_state=t["has_initial_state"],
                                      act=act, dev_status=status)
    torch.cuda.synchronize()
    y_ref, p_ref = oracle.conv_prefill(d["x"], d["w"], d["cu_seqlens"], d["state_indices"], d["pool"],
                                       bias=d["b"], has_initial_state=d["has_initial_state"], act=act)
    assert int(status.item()) == 0
    tol = 1e-5 if dtype == torch.float32 else 1e-3
    assert excess_error(y, y_ref) <= tol
    assert excess_error(t["pool"], p_ref) <= 0.0 + (1e-6 if dtype == torch.float32 else 0.0)
    t0, t1 = int(d["cu_seqlens"][8]), int(d["cu_seqlens"][9])
    assert torch.count_nonzero(y[t0:t1].float()).item() == 0  # padding rows exactly zero
    used = set(int(i) for i in idx.tolist() if i >= 0)
    for s_ in range(16):
        if s_ not in used:
            assert torch.equal(t["pool"][s_].cpu(), d["pool"][s_])


def test_conv_prefill_many_sequences(kda_gpu):
    """70 sequences of 0-130 tokens (more than one 32-sequence lookup step)."""
    gen = torch.Generator().manual_seed(71)
    lens = tuple(int(x) for x in torch.randint(0, 131, (70,), generator=gen))
    d = W_.make_conv(lens, 264, 4, torch.bfloat16, num_slots=80, seed=72)
    t = to_dev(d, DEV)
    y = torch.full_like(t["x"], float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda_gpu.kda_causal_conv1d_prefill(t["x"], t["w"], t["cu_seqlens"], t["state_indices"], t["pool"],
                                      y, bias=t["b"], dev_status=status)
    torch.cuda.synchronize()
    y_ref, p_ref = oracle.conv_prefill(d["x"], d["w"], d["cu_seqlens"], d["state_indices"], d["pool"],
                                       bias=d["b"])
    assert int(status.item()) == 0
    assert excess_error(y, y_ref) <= 1e-3
    assert excess_error(t["pool"], p_ref) <= 0.0


@pytest.mark.parametrize("dtype,W", [(torch.bfloat16, 4), (torch.float32, 3)])
def test_conv_prefill_many_items_per_cta(kda_gpu, dtype, W):
    """The scheduler's 8-sequence mix (4096 tokens) over 12288 channels: several
    thousand (tile, channel block) items, so every CTA of the persistent grid
    takes many in turn; one sequence without initial state, one padding."""
    lens = (1576, 586, 148, 147, 122, 303, 788, 426)
    his = [1, 0, 1, 1, 1, 1, 1, 1]
    d = W_.make_conv(lens, 12288, W, dtype, num_slots=12, seed=1234 + W, has_initial=his)
    idx = d["state_indices"].clone()
    idx[4] = -1
    d["state_indices"] = idx
    t = to_dev(d, DEV)
    y = torch.full_like(t["x"], float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda_gpu.kda_causal_conv1d_prefill(t["x"], t["w"], t["cu_seqlens"], t["state_indices"], t["pool"],
                                      y, bias=t["b"], has_initial_state=t["has_initial_state"],
                                      dev_status=status)
    torch.cuda.synchronize()
    y_ref, p_ref = oracle.conv_prefill(d["x"], d["w"], d["cu_seqlens"], d["state_indices"], d["pool"],
                                       bias=d["b"], has_initial_state=d["has_initial_state"])
    assert int(status.item()) == 0
    tol = 1e-5 if dtype == torch.float32 else 1e-3
    assert excess_error(y, y_ref) <= tol
    assert excess_error(t["pool"], p_ref) <= (1e-6 if dtype == torch.float32 else 0.0)


def _check_prefill_conv(kda, w, d, conv_act, *, label=None):
    """The fused convolution + normalisation + prefill against the oracle's
    pipeline: outputs, states and checkpoints within the tolerance rule, the
    convolution cache bit-exact (its rows are copies of inputs), checkpoint
    offsets exact, untouched slots of both pools unchanged."""
    pool0, cpool0 = d["pool"].clone(), d["conv_pool"].clone()
    out, pool, ck, offs, status, cpool = run_prefill_conv(kda, d, w, DEV, conv_act=conv_act)
    assert int(status.item()) == 0, kda.DEV_STATUS[int(status.item())]
    o_ref, p_ref, ck_ref, offs_ref, c_ref = oracle_prefill_conv(oracle, d, w, conv_act=conv_act)
    tol = tol_for(w.state_dtype)
    if label:
        record(label, "out", out, o_ref)
    assert excess_error(out, o_ref) <= tol
    idx = d["state_indices"].tolist()
    lens = (d["cu_seqlens"][1:] - d["cu_seqlens"][:-1]).tolist()
    touched = [s for s, L in zip(idx, lens) if s >= 0 and L > 0]
    pool_cpu, cpool_cpu = pool.cpu(), cpool.cpu()
    for s in range(w.num_slots):
        if s in touched:
            if label:
                record(label, "final_state", pool_cpu[s], p_ref[s])
            assert excess_error(pool_cpu[s], p_ref[s]) <= tol, s
            assert np.array_equal(cpool_cpu[s].double().numpy(), c_ref[s]), f"conv cache of slot {s}"
        else:
            assert torch.equal(pool_cpu[s], pool0[s]), f"slot {s} modified"
            assert torch.equal(cpool_cpu[s], cpool0[s]), f"conv cache of slot {s} modified"
    if w.checkpoint_every:
        assert offs.cpu().numpy().tolist() == offs_ref.tolist()
        real = []
        for i, s in enumerate(idx):
            if s >= 0:
                real.extend(range(int(offs_ref[i]), int(offs_ref[i + 1])))
        if real:
            assert excess_error(ck[real], ck_ref[real]) <= tol
    for i, s in enumerate(idx):
        if s < 0:  # padding rows exactly zero
            t0, t1 = int(d["cu_seqlens"][i]), int(d["cu_seqlens"][i + 1])
            assert torch.count_nonzero(out[t0:t1].float()).item() == 0
    return out


@pytest.mark.parametrize("d,cw,act,state_dtype", [(128, 4, "silu", torch.float32),
                                                  (128, 3, "none", torch.bfloat16),
                                                  (64, 2, "silu", torch.float32),
                                                  (64, 4, "silu", torch.bfloat16)])
def test_prefill_conv_fused(kda_gpu, d, cw, act, state_dtype):
    """Convolution widths 2-4 and both activations in front of the tensor-core
    prefill: lengths shorter than the convolution's context (the cache keeps
    old rows), chunk edges, an empty and a padding sequence, a mix of
    initial-state flags (the flag governs both the state and the convolution
    cache), gate, checkpoints every 64 tokens."""
    lens = (1, 2, 3, 63, 64, 65, 0, 200, 130, 5)
    w = W.SCHED.replace(seqlens=lens, H=4, dk=d, dv=d, num_slots=14, slot_range=None,
                        state_dtype=state_dtype, checkpoint_every=64, seed=900 + d + cw)
    inp = W.make_prefill_conv(w, cw)
    inp["state_indices"][8] = -1
    inp["has_initial_state"] = torch.tensor([1, 0, 1, 1, 0, 1, 1, 1, 0, 1], dtype=torch.int32)
    _check_prefill_conv(kda_gpu, w, inp, act)


def test_prefill_conv_fused_many_sequences(kda_gpu):
    """70 sequences of 0-130 tokens (the chunk lookup steps past 32 sequences;
    many are shorter than the convolution's context), width 3, d = 64, bf16
    state, a mix of initial-state flags and two padding sequences."""
    gen = torch.Generator().manual_seed(951)
    lens = [int(x) for x in torch.randint(0, 131, (70,), generator=gen)]
    lens[3], lens[40] = 1, 2
    w = W.VARLEN.replace(seqlens=tuple(lens), H=2, dk=64, dv=64, num_slots=80, state_dtype=torch.bfloat16,
                         checkpoint_every=64, seed=952)
    d = W.make_prefill_conv(w, 3)
    d["state_indices"][[10, 55]] = -1
    d["has_initial_state"] = (torch.arange(70) % 3 != 0).to(torch.int32)
    _check_prefill_conv(kda_gpu, w, d, "silu")


def test_prefill_conv_fused_sched_workload(kda_gpu):
    """The 4096-token scheduler mix at its full width (32 heads of 128) with a
    width-4 SiLU convolution in front, with the output norm-gate and without
    it (the ungated output shows the error before the norm's division by
    rms(o) amplifies the rare bf16 rounding flips of the intermediate q/k/v)."""
    w = W.SCHED
    _check_prefill_conv(kda_gpu, w, W.make_prefill_conv(w, 4), "silu", label=w.name + "_conv4")
    wu = w.replace(gate=False)
    out = _check_prefill_conv(kda_gpu, wu, W.make_prefill_conv(wu, 4), "silu", label=w.name + "_conv4_nogate")
    assert out.shape == (w.T, w.H, w.dv)


def test_prefill_conv_fused_equals_the_separate_calls(kda_gpu):
    """The fused call against the three library calls it replaces, run one
    after another on the same inputs (convolution, L2 normalisation in torch
    on the device with bf16 rounding, prefill): the convolution caches agree
    bit for bit and the outputs within the tolerance."""
    w = W.VARLEN.replace(dk=128, dv=128, H=4, seqlens=(3, 100, 64, 129), num_slots=8, seed=931)
    d = W.make_prefill_conv(w, 4)
    out_f, pool_f, _, _, status, cpool_f = run_prefill_conv(kda_gpu, d, w, DEV, ckpt=False)
    assert int(status.item()) == 0
    t = to_dev(d, DEV)
    T = t["x"].shape[0]
    y = torch.empty_like(t["x"])
    kda_gpu.kda_causal_conv1d_prefill(t["x"], t["conv_w"], t["cu_seqlens"], t["state_indices"], t["conv_pool"],
                                      y, bias=t["conv_b"], act="silu")
    yq, yk, yv = (y.reshape(T, 3, w.H, w.dk)[:, i].float() for i in range(3))
    nq = (yq / torch.sqrt((yq * yq).sum(-1, keepdim=True) + 1e-6)).to(w.in_dtype).contiguous()
    nk = (yk / torch.sqrt((yk * yk).sum(-1, keepdim=True) + 1e-6)).to(w.in_dtype).contiguous()
    sep = dict(d, q=nq, k=nk, v=yv.to(w.in_dtype).contiguous())
    sep = {k: v for k, v in sep.items() if k not in ("x", "conv_w", "conv_b", "conv_pool")}
    sep["pool"] = d["pool"].clone()
    out_s, pool_s, _, _, status = run_prefill(kda_gpu, sep, w, DEV, ckpt=False)
    assert int(status.item()) == 0
    assert torch.equal(cpool_f, t["conv_pool"])
    assert (out_f.float() - out_s.float()).abs().max().item() <= 0.01
    assert (pool_f - pool_s).abs().max().item() <= 0.01


def test_prefill_conv_bad_conv_slot_latches_status(kda_gpu):
    """An index inside the state pool but past the convolution pool latches
    the bad-index status; that sequence's rows are zero and no slot changes."""
    w = W.VARLEN.replace(dk=64, dv=64, H=2, seqlens=(70, 30), num_slots=6, seed=937)
    d = W.make_prefill_conv(w, 3)
    d["conv_pool"] = d["conv_pool"][:4].contiguous()
    d["state_indices"] = torch.tensor([1, 5], dtype=torch.int32)
    pool0, cpool0 = d["pool"].clone(), d["conv_pool"].clone()
    out, pool, _, _, status, cpool = run_prefill_conv(kda_gpu, d, w, DEV, ckpt=False)
    assert int(status.item()) == 1
    assert torch.count_nonzero(out[70:].float()).item() == 0
    assert torch.equal(pool[5].cpu(), pool0[5])
    assert torch.equal(cpool.cpu()[[0, 2, 3]], cpool0[[0, 2, 3]])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_conv_decode_steps_and_split(kda_gpu, dtype):
    """A prefill of 40 tokens then 6 decode steps equals the oracle's prefill of
    all 46 tokens (outputs and final cache), over a 12288-channel (3 x 32 x 128)
    projection."""
    C, W = 12288, 4
    lens = (40, 17)
    d = W_.make_conv(lens, C, W, dtype, num_slots=4, seed=91)
    extra = torch.randn(6, 2, C, generator=torch.Generator().manual_seed(5)).to(dtype)
    t = to_dev(d, DEV)
    y = torch.empty_like(t["x"])
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda_gpu.kda_causal_conv1d_prefill(t["x"], t["w"], t["cu_seqlens"], t["state_indices"], t["pool"],
                                      y, bias=t["b"], dev_status=status)
    ys = []
    for s_ in range(6):
        xs = extra[s_].to(DEV)
        ysd = torch.empty_like(xs)
        kda_gpu.kda_causal_conv1d_decode(xs, t["w"], t["state_indices"], t["pool"], ysd, bias=t["b"],
                                         dev_status=status)
        ys.append(ysd)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # the oracle over the concatenated sequences
    xa = torch.cat([d["x"][:40], extra[:, 0], d["x"][40:], extra[:, 1]])
    cua = torch.tensor([0, 46, 46 + 23], dtype=torch.int32)
    y_ref, p_ref = oracle.conv_prefill(xa, d["w"], cua, d["state_indices"], d["pool"], bias=d["b"])
    tol = 1e-5 if dtype == torch.float32 else 1e-3
    assert excess_error(y[:40], y_ref[:40]) <= tol
    assert excess_error(y[40:], y_ref[46:63]) <= tol
    dec = torch.stack(ys)  # [6, 2, C]
    assert excess_error(dec[:, 0], y_ref[40:46]) <= tol
    assert excess_error(dec[:, 1], y_ref[63:69]) <= tol
    assert excess_error(t["pool"], p_ref) <= (1e-6 if dtype == torch.float32 else 0.0)


@pytest.mark.parametrize("dv", [16, 64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("variant", ["residual_prenorm", "bias_no_weight", "packed_gate",
                                     "in_place"])
def test_norm_gate_variants(kda_gpu, dv, dtype, variant):
    """The norm-gate variants against the oracle: residual with prenorm output,
    bias without weight (SiLU), a gate read from a packed projection row, and
    in-place outputs (y over o, prenorm over residual)."""
    gen = torch.Generator().manual_seed(500 + dv)
    rows, H = 29, 3
    mk = lambda *sh: torch.randn(*sh, generator=gen).to(dtype)
    o, res, gate = mk(rows, H, dv), mk(rows, H, dv), mk(rows, H, dv)
    w = (1 + 0.05 * torch.randn(dv, generator=gen)).to(dtype)
    b = (0.2 * torch.randn(dv, generator=gen)).to(dtype)
    act = "silu" if variant == "bias_no_weight" else "sigmoid"
    use_res = variant in ("residual_prenorm", "in_place")
    use_w = variant != "bias_no_weight"
    use_b = variant in ("bias_no_weight", "residual_prenorm")
    if variant == "packed_gate":
        packed = mk(rows, H * dv + 32)
        packed[:, 16:16 + H * dv] = gate.reshape(rows, -1)
        dpacked = packed.to(DEV)
        dgate = dpacked[:, 16:16 + H * dv].view(rows, H, dv)
    else:
        dgate = gate.to(DEV)
    y_ref, x_ref = oracle.norm_gate_ex(o, gate, residual=res if use_res else None,
                                       w=w if use_w else None, b=b if use_b else None, eps=1e-6,
                                       gate_act=act)
    od, rd = o.to(DEV), res.to(DEV)
    y = od if variant == "in_place" else torch.empty_like(od)
    rout = rd if variant == "in_place" else (torch.empty_like(od) if use_res else None)
    kda_gpu.kda_norm_gate_ex(od, dgate, y, residual=rd if use_res else None, residual_out=rout,
                             w=w.to(DEV) if use_w else None, b=b.to(DEV) if use_b else None,
                             eps=1e-6, gate_act=act)
    torch.cuda.synchronize()
    tol = 1e-5 if dtype == torch.float32 else 1e-3
    assert excess_error(y, y_ref) <= tol
    if rout is not None:
        assert excess_error(rout, x_ref) <= tol
    if variant != "in_place":
        assert torch.equal(od.cpu(), o)  # inputs preserved
        assert torch.equal(rd.cpu(), res)
    if variant == "packed_gate":
        assert torch.equal(dpacked.cpu(), packed)  # the rest of the packed row untouched


@pytest.mark.parametrize("dv", [16, 64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("inplace", [False, True])
@pytest.mark.parametrize("act", ["sigmoid", "silu"])
def test_norm_gate(kda_gpu, dv, dtype, inplace, act):
    gen = torch.Generator().manual_seed(dv)
    o = torch.randn(37, 5, dv, generator=gen).to(dtype)
    gate = torch.randn(37, 5, dv, generator=gen).to(dtype)
    w = (1 + 0.02 * torch.randn(dv, generator=gen)).to(dtype)
    ref = oracle.norm_gate(o, gate, w, eps=1e-6, gate_act=act)
    od, gd, wd = o.to(DEV), gate.to(DEV), w.to(DEV)
    y = od if inplace else torch.empty_like(od)
    kda_gpu.kda_norm_gate(od, gd, wd, y, eps=1e-6, gate_act=act)
    torch.cuda.synchronize()
    assert excess_error(y, ref) <= 1e-5 if dtype == torch.float32 else excess_error(y, ref) <= 1e-2
    if not inplace:
        assert torch.equal(od.cpu(), o)  # input preserved


def test_binding_rejects_mismatched_arguments(kda_gpu):
    """A size that disagrees with q, an int64 index array or a host tensor among
    device tensors raise ValueError in the binding; nothing is launched."""
    w = W.VARLEN
    d = W.make_prefill(w)
    t = to_dev(d, DEV)
    T = t["q"].shape[0]
    out = torch.full((T, w.H, w.dv), 7.0, device=DEV, dtype=w.in_dtype)
    ws = torch.empty(kda_gpu.kda_prefill_workspace_bytes(w.N, T, w.H, w.dk, w.dv, w.chunk) + 16,
                     dtype=torch.uint8, device=DEV)

    def call(**over):
        a = dict(t, out=out)
        a.update(over)
        kda_gpu.kda_prefill_chunked(a["q"], a["k"], a["v"], a["g"], a["beta"], a["cu_seqlens"],
                                    a["state_indices"], a["pool"], a["out"], chunk=w.chunk,
                                    workspace=ws)

    with pytest.raises(ValueError, match="k must have shape"):
        call(k=t["k"][:-1])
    with pytest.raises(ValueError, match="state_indices must be torch.int32"):
        call(state_indices=t["state_indices"].long())
    with pytest.raises(ValueError, match="one CUDA device"):
        call(beta=d["beta"])
    with pytest.raises(ValueError, match="out must have shape"):
        call(out=out[:, :, :-1].contiguous())
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())  # nothing ran


@pytest.mark.parametrize("dim", [64, 128])
def test_graph_capture_replay(kda_gpu, dim):
    """A prefill and a decode step captured in one CUDA graph and replayed give
    the eager results (the ABI makes no host sync or host read)."""
    w = W.VARLEN.replace(dk=dim, dv=dim)
    d = W.make_prefill(w)
    t = to_dev(d, DEV)
    out = torch.empty(w.T, w.H, w.dv, device=DEV, dtype=w.in_dtype)
    wsb = kda_gpu.kda_prefill_workspace_bytes(w.N, w.T, w.H, w.dk, w.dv, w.chunk)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=DEV)
    pool_init = t["pool"].clone()
    dw = W.DECODE.replace(N=4, H=w.H, dk=w.dk, dv=w.dv, num_slots=w.num_slots)
    sd = to_dev(W.make_decode_step(dw, 0), DEV)
    dout = torch.empty(dw.N, dw.H, dw.dv, device=DEV, dtype=dw.in_dtype)
    didx = torch.tensor([0, 5, 9, 15], dtype=torch.int32, device=DEV)
    nw = torch.ones(w.dv, device=DEV, dtype=w.in_dtype)

    def step(stream=None):
        kda_gpu.kda_prefill_chunked(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"],
                                    t["state_indices"], t["pool"], out, chunk=w.chunk,
                                    scale=d["scale"], workspace=ws, stream=stream)
        kda_gpu.kda_decode_step(sd["q"], sd["k"], sd["v"], sd["g"], sd["beta"], didx, t["pool"],
                                dout, gate=sd["gate"], norm_w=nw, stream=stream)

    step()
    torch.cuda.synchronize()
    out_e, dout_e, pool_e = out.clone(), dout.clone(), t["pool"].clone()
    t["pool"].copy_(pool_init)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            step(stream=s)
    torch.cuda.synchronize()
    t["pool"].copy_(pool_init)
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, out_e) and torch.equal(dout, dout_e) and torch.equal(t["pool"], pool_e)


def test_graph_capture_replay_conv_fused(kda_gpu):
    """The fused convolution prefill captured in a CUDA graph, gated and with
    checkpoints: one replay equals an eager call, and a second replay carries
    both pools updated in place (the recurrent state and the convolution cache)
    exactly like a second eager call.  The first sequence is shorter than the
    convolution's context, so its cache keeps old rows and moves on with every
    call."""
    w = W.VARLEN.replace(dk=128, dv=128, H=4, seqlens=(2, 100, 64, 129), num_slots=8,
                         checkpoint_every=64, gate=True, seed=961)
    d = W.make_prefill_conv(w, 4)
    t = to_dev(d, DEV)
    T = t["x"].shape[0]
    out = torch.empty(T, w.H, w.dv, device=DEV, dtype=w.in_dtype)
    ck = torch.zeros(T // 64, w.H, w.dk, w.dv, device=DEV, dtype=w.state_dtype)
    offs = torch.zeros(w.N + 1, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    wsb = kda_gpu.kda_prefill_workspace_bytes(w.N, T, w.H, w.dk, w.dv, w.chunk)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=DEV)
    pool0, cpool0 = t["pool"].clone(), t["conv_pool"].clone()

    def step(stream=None):
        kda_gpu.kda_prefill_chunked_conv(t["x"], t["conv_w"], t["conv_pool"], t["g"], t["beta"],
                                         t["cu_seqlens"], t["state_indices"], t["pool"], out,
                                         conv_b=t["conv_b"], conv_act="silu", chunk=w.chunk,
                                         checkpoints=ck, checkpoint_every=64, ckpt_offsets=offs,
                                         gate=t["gate"], norm_w=t["norm_w"], eps=d.get("eps", 1e-6),
                                         scale=d["scale"], workspace=ws, dev_status=status,
                                         stream=stream)

    eager = []
    for _ in range(2):
        step()
        torch.cuda.synchronize()
        eager.append((out.clone(), t["pool"].clone(), t["conv_pool"].clone(), ck.clone()))
    assert int(status.item()) == 0
    slot = int(d["state_indices"][0])
    assert not torch.equal(eager[0][2][slot], eager[1][2][slot])  # the second call moved that cache on
    t["pool"].copy_(pool0)
    t["conv_pool"].copy_(cpool0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            step(stream=s)
    torch.cuda.synchronize()
    t["pool"].copy_(pool0)
    t["conv_pool"].copy_(cpool0)
    for i in range(2):
        out.zero_()
        ck.zero_()
        graph.replay()
        torch.cuda.synchronize()
        o_e, p_e, c_e, k_e = eager[i]
        assert torch.equal(out, o_e) and torch.equal(t["pool"], p_e), i
        assert torch.equal(t["conv_pool"], c_e) and torch.equal(ck, k_e), i
    assert int(status.item()) == 0
