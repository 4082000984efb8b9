"""GPU parity at pool slots whose element offsets pass 2^31.

With H = 32 and d = 128 a state slot holds 2^19 elements, so in an fp32 pool
every slot from 4096 on starts beyond element 2^31; the convolution cache
[slots, W-1, C] with C = 12288 and W = 4 passes it from slot 58255 on.  The
pools here are that large on the device (8.8 GB and 4.4 GB), but only the
touched slots and a few untouched neighbours are ever written from the host.
The oracle runs on the touched slots alone, remapped to a small pool: every
state and cache value, every output and checkpoint against it, and the
neighbours bit-identical afterwards.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from kda_testutil import excess_error, oracle_prefill, tol_for

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")

H, D = 32, 128
STATE_SLOTS = 4200                  # 4200 x 32 x 128 x 128 x 4 B = 8.8 GB
STATE_BIG = [4199, 4096, 17]        # small-pool slot j lives at STATE_BIG[j]
STATE_NEIGHBOURS = [4198, 4097, 4095, 18]


def _big_pool(small, big_slots, total, neighbours, dtype):
    """A device pool of `total` slots with small[j] at big_slots[j] and a
    seeded pattern in the neighbour slots (the rest is left unwritten)."""
    pool = torch.empty((total,) + tuple(small.shape[1:]), device=DEV, dtype=dtype)
    for j, s in enumerate(big_slots):
        pool[s] = small[j].to(DEV)
    gen = torch.Generator().manual_seed(4242)
    marks = {s: torch.randn(tuple(small.shape[1:]), generator=gen).to(dtype) for s in neighbours}
    for s, m in marks.items():
        pool[s] = m.to(DEV)
    return pool, marks


def _neighbours_intact(pool, marks):
    for s, m in marks.items():
        assert torch.equal(pool[s].cpu(), m), f"slot {s} modified"


def test_state_pool_beyond_2_31_elements(kda_gpu):
    """Prefill (tensor-core path, checkpoints, gate), a decode step, then a
    3-token verification with its commit, all on slots 4199, 4096 and 17 of an
    8.8 GB fp32 pool."""
    w = W.PrefillWorkload("large_offsets", (100, 64, 37), H, D, D, 64, 64, torch.bfloat16,
                          torch.float32, 3, True, False, 61)
    d = W.make_prefill(w)
    small_idx = d["state_indices"]                       # a permutation of 0..2
    big_idx = torch.tensor([STATE_BIG[int(j)] for j in small_idx], dtype=torch.int32)
    pool, marks = _big_pool(d["pool"], STATE_BIG, STATE_SLOTS, STATE_NEIGHBOURS, torch.float32)
    t = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    T = int(d["cu_seqlens"][-1])
    I = w.checkpoint_every
    ck = torch.full((T // I, H, D, D), float("nan"), device=DEV)
    offs = torch.zeros(len(w.seqlens) + 1, dtype=torch.int32, device=DEV)
    out = torch.full((T, H, D), float("nan"), device=DEV, dtype=torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(kda_gpu.kda_prefill_workspace_bytes(3, T, H, D, D, 64), dtype=torch.uint8,
                     device=DEV)
    kda_gpu.kda_prefill_chunked(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"],
                                big_idx.to(DEV), pool, out, chunk=64, checkpoints=ck,
                                checkpoint_every=I, ckpt_offsets=offs, gate=t["gate"],
                                norm_w=t["norm_w"], eps=d["eps"], scale=d["scale"], workspace=ws,
                                dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o_ref, p_ref, ck_ref, offs_ref = oracle_prefill(oracle, d, w)
    tol = tol_for(torch.float32)
    assert excess_error(out, o_ref) <= tol
    assert offs.cpu().tolist() == offs_ref.tolist()
    n_ck = int(offs_ref[-1])
    assert excess_error(ck[:n_ck], ck_ref[:n_ck]) <= tol
    for j, s in enumerate(STATE_BIG):
        assert excess_error(pool[s], p_ref[j]) <= tol, s
    _neighbours_intact(pool, marks)

    # one decode step on the same slots (small slot j at STATE_BIG[j])
    dw = W.DECODE.replace(N=3, num_slots=3, seed=62)
    step = W.make_decode_step(dw, 0)
    nw = t["norm_w"]
    sd = {k: v.to(DEV) for k, v in step.items()}
    idx_small = torch.arange(3, dtype=torch.int32)
    idx_big = torch.tensor(STATE_BIG, dtype=torch.int32, device=DEV)
    y = torch.full((3, H, D), float("nan"), device=DEV, dtype=torch.bfloat16)
    kda_gpu.kda_decode_step(sd["q"], sd["k"], sd["v"], sd["g"], sd["beta"], idx_big, pool, y,
                            gate=sd["gate"], norm_w=nw, eps=d["eps"], dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    y_ref, p_dec = oracle.decode(step["q"], step["k"], step["v"], step["g"], step["beta"],
                                 idx_small, p_ref, gate=step["gate"], norm_w=d["norm_w"],
                                 eps=d["eps"])
    assert excess_error(y, y_ref) <= tol
    for j, s in enumerate(STATE_BIG):
        assert excess_error(pool[s], p_dec[j]) <= tol, s

    # 3 draft tokens per sequence, then the commit of 3, 0 and 2 accepted tokens
    K = 3
    dr = W.make_decode_draft(dw, K)
    dr.pop("num_accepted")
    acc = torch.tensor([3, 0, 2], dtype=torch.int32)
    dd = {k: v.to(DEV) for k, v in dr.items()}
    ym = torch.full((3, K, H, D), float("nan"), device=DEV, dtype=torch.bfloat16)
    ts = torch.full((3, K, H, D, D), float("nan"), device=DEV)
    kda_gpu.kda_decode_multi(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], idx_big, pool, ym, ts,
                             gate=dd["gate"], norm_w=nw, eps=d["eps"], dev_status=status)
    kda_gpu.kda_commit_accepted(ts, acc.to(DEV), idx_big, pool, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ym_ref, ts_ref, _ = oracle.decode_multi(dr["q"], dr["k"], dr["v"], dr["g"], dr["beta"],
                                            idx_small, p_dec, gate=dr["gate"],
                                            norm_w=d["norm_w"], eps=d["eps"])
    p_commit = oracle.commit_accepted(ts_ref, acc.numpy(), idx_small.numpy(), p_dec)
    assert excess_error(ym, ym_ref) <= tol
    assert excess_error(ts, ts_ref) <= tol
    for j, s in enumerate(STATE_BIG):
        assert excess_error(pool[s], p_commit[j]) <= tol, s
    _neighbours_intact(pool, marks)


CONV_SLOTS = 60000                   # 60000 x 3 x 12288 x 2 B = 4.4 GB
CONV_BIG = [59999, 58255, 3]
CONV_NEIGHBOURS = [59998, 58254, 58256, 4]


def test_conv_cache_pool_beyond_2_31_elements(kda_gpu):
    """The convolution prefill and two decode steps on cache slots 59999, 58255
    and 3 of a [60000, 3, 12288] bf16 cache pool."""
    C, Wd = 12288, 4
    d = W.make_conv((70, 5, 1), C, Wd, torch.bfloat16, num_slots=3, seed=63,
                    has_initial=[1, 0, 1])
    small_idx = d["state_indices"]
    big_idx = torch.tensor([CONV_BIG[int(j)] for j in small_idx], dtype=torch.int32)
    pool, marks = _big_pool(d["pool"], CONV_BIG, CONV_SLOTS, CONV_NEIGHBOURS, torch.bfloat16)
    t = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    y = torch.full_like(t["x"], float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda_gpu.kda_causal_conv1d_prefill(t["x"], t["w"], t["cu_seqlens"], big_idx.to(DEV), pool, y,
                                      bias=t["b"], has_initial_state=t["has_initial_state"],
                                      dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    y_ref, p_ref = oracle.conv_prefill(d["x"], d["w"], d["cu_seqlens"], small_idx, d["pool"],
                                       bias=d["b"], has_initial_state=d["has_initial_state"])
    assert excess_error(y, y_ref) <= 1e-3
    for j, s in enumerate(CONV_BIG):
        assert excess_error(pool[s], p_ref[j]) <= 0.0, s
    _neighbours_intact(pool, marks)
    gen = torch.Generator().manual_seed(64)
    idx_small = torch.arange(3, dtype=torch.int32)
    idx_big = torch.tensor(CONV_BIG, dtype=torch.int32, device=DEV)
    ref_pool = p_ref
    for _ in range(2):
        x1 = torch.randn(3, C, generator=gen).to(torch.bfloat16)
        y1 = torch.full((3, C), float("nan"), device=DEV, dtype=torch.bfloat16)
        kda_gpu.kda_causal_conv1d_decode(x1.to(DEV), t["w"], idx_big, pool, y1, bias=t["b"],
                                         dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        y1_ref, ref_pool = oracle.conv_decode(x1, d["w"], idx_small, ref_pool, bias=d["b"])
        assert excess_error(y1, y1_ref) <= 1e-3
    for j, s in enumerate(CONV_BIG):
        assert excess_error(pool[s], ref_pool[j]) <= 0.0, s
    _neighbours_intact(pool, marks)
