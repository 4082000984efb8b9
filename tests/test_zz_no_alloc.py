"""The prefill entry point for callers that cannot allocate device memory
(kda_prefill_chunked_static_scratch): it must give what kda_prefill_chunked
gives with a caller-allocated workspace, on consecutive calls that reuse the
library's one scratch array, and must refuse sizes beyond that array.

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test."""
import pytest
import torch

import workloads as W
from kda_testutil import excess_error, max_abs, to_dev, tol_for

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _run(kda, d, w, pool, *, static, ws=None):
    t = to_dev(d, DEV)
    out = torch.empty(w.T, w.H, w.dv, device=DEV, dtype=w.in_dtype)
    ck = torch.empty(w.T // w.checkpoint_every, w.H, w.dk, w.dv, device=DEV, dtype=w.state_dtype)
    offs = torch.empty(w.N + 1, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    args = (t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"], t["state_indices"], pool, out)
    kw = dict(chunk=w.chunk, checkpoints=ck, checkpoint_every=w.checkpoint_every, ckpt_offsets=offs,
              gate=t["gate"], norm_w=t["norm_w"], eps=d["eps"], scale=d["scale"], dev_status=status)
    if static:
        kda.kda_prefill_chunked_static_scratch(*args, **kw)
    else:
        kda.kda_prefill_chunked(*args, workspace=ws, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out, ck, offs


def test_static_scratch_matches_workspace_entry_point(kda_gpu):
    kda = kda_gpu
    import oracle
    # tensor-core shape; its scratch fits the array
    w = W.SCHED.replace(seqlens=(300, 100, 700), H=8, num_slots=16, slot_range=None,
                        checkpoint_every=128, seed=501)
    need = kda.kda_prefill_workspace_bytes(w.N, w.T, w.H, w.dk, w.dv, w.chunk)
    assert 0 < need <= kda.STATIC_SCRATCH_BYTES
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    pool0 = W.make_prefill(w)["pool"]
    pool_ref, pool_static = pool0.to(DEV), pool0.to(DEV)
    pool_oracle = pool0.double().numpy()
    tol = tol_for(w.state_dtype)
    for call in range(2):  # consecutive calls carry the state and reuse the scratch
        d = W.make_prefill(w, seed=w.seed + call)
        o_ref, ck_ref, off_ref = _run(kda, d, w, pool_ref, static=False, ws=ws)
        o_st, ck_st, off_st = _run(kda, d, w, pool_static, static=True)
        written = int(off_ref[-1].item())  # entries past the last offset are never written
        assert written == 7
        # the same kernels on the same inputs: identical bits, whichever scratch they use
        assert torch.equal(o_st, o_ref)
        assert torch.equal(ck_st[:written], ck_ref[:written])
        assert torch.equal(pool_static, pool_ref)
        assert torch.equal(off_st, off_ref)
        # and both within the bound of the fp64 oracle carried through the same calls
        d["pool"] = pool_oracle
        y, pool_oracle, ck, offs = oracle.prefill(
            d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["state_indices"],
            d["pool"], checkpoint_every=w.checkpoint_every, gate=d["gate"], norm_w=d["norm_w"],
            eps=d["eps"], scale=d["scale"])
        assert excess_error(o_st, y) <= tol
        assert max_abs(ck_st[:written], ck) <= tol
        assert max_abs(pool_static, pool_oracle) <= tol
        assert off_st.cpu().tolist() == list(offs)


def test_static_scratch_rejects_oversize(kda_gpu):
    kda = kda_gpu
    lib = kda.load()
    fake = 1 << 20  # never dereferenced: the size check comes first
    # 65536 tokens x 32 heads needs ~2.4 GB of scratch, far above the array
    rc = lib.kda_prefill_chunked_static_scratch(
        fake, fake, fake, fake, fake, 1, fake, 1, 65536, fake, None, fake, 4, 0, fake, None, 0, 0,
        None, None, None, 1e-6, 0, 32, 128, 128, 64, 0.0, None, None)
    assert rc == -3  # KDA_ERR_WORKSPACE
