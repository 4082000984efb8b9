"""A bounded on-chip wait that runs out.  With the testing hook set to zero
polls, the first wait of the selected tensor-core prefill kernel gives up at
once.  The call must still return and report KDA_DEV_TIMEOUT (3) instead of
hanging or trapping, and nothing may be written to the pool:
  * intra-chunk kernel: every CTA gives up and stamps its workspace block
    failed; the state kernel, whose own waits succeed, must see the stamps
    and store nothing (no stale workspace data carried into the pool);
  * state kernel: every chain gives up on its first operand copy and drains
    the copies and products still in flight before it exits;
  * both.
After the hook is reset, the next call on the same stream must match the
oracle.  With the short convolution fused in, a chain that gives up also
leaves its slot's convolution cache as it was: a failed sequence is skipped,
its recurrent state and convolution cache together.

Nothing here makes the GPU fault: a wait gives up on its own count, and the
kernels' clean-up lets every bulk copy and tensor-core product in flight
finish before their shared and tensor memory are released."""
import pytest
import torch

import oracle
import workloads as W
from kda_testutil import (excess_error, max_abs, oracle_prefill, oracle_prefill_conv, run_prefill,
                          run_prefill_conv, tol_for)

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.mark.parametrize("kernels", [1, 2, 3], ids=["intra", "state", "both"])
def test_first_wait_timeout_reports_and_recovers(kda_gpu, kernels):
    kda = kda_gpu
    w = W.SCHED.replace(seqlens=(150, 64, 1), H=4, num_slots=8, slot_range=None,
                        checkpoint_every=64, seed=808)
    d = W.make_prefill(w)
    pool0 = d["pool"].clone()
    try:
        kda.kda_testing_set_first_wait_tries(0, kernels)
        out, pool, ck, offs, status = run_prefill(kda, d, w, DEV)
        assert int(status.item()) == 3, kda.DEV_STATUS.get(int(status.item()))
        # every state chain stopped before its first product: no slot written
        assert torch.equal(pool.cpu(), pool0)
    finally:
        kda.kda_testing_set_first_wait_tries(-1)
    # the same call again, limits back to normal, on a fresh status word
    d2 = dict(d, pool=pool0.clone())
    out, pool, ck, offs, status = run_prefill(kda, d2, w, DEV)
    assert int(status.item()) == 0
    o_ref, p_ref, ck_ref, offs_ref = oracle_prefill(oracle, d2, w)
    tol = tol_for(w.state_dtype)
    assert excess_error(out, o_ref) <= tol
    touched = d["state_indices"].long().tolist()
    assert max_abs(pool[touched], p_ref[touched]) <= tol
    assert offs.cpu().tolist() == offs_ref.tolist()
    n = int(offs_ref[-1])
    assert max_abs(ck[:n], ck_ref[:n]) <= tol


@pytest.mark.parametrize("kernels", [1, 2, 3], ids=["intra", "state", "both"])
def test_first_wait_timeout_conv_fused_keeps_both_pools(kda_gpu, kernels):
    kda = kda_gpu
    w = W.SCHED.replace(seqlens=(150, 64, 1), H=4, num_slots=8, slot_range=None,
                        checkpoint_every=64, seed=809)
    d = W.make_prefill_conv(w, 4)
    pool0, cpool0 = d["pool"].clone(), d["conv_pool"].clone()
    try:
        kda.kda_testing_set_first_wait_tries(0, kernels)
        out, pool, ck, offs, status, cpool = run_prefill_conv(kda, d, w, DEV)
        assert int(status.item()) == 3, kda.DEV_STATUS.get(int(status.item()))
        assert torch.equal(pool.cpu(), pool0)
        assert torch.equal(cpool.cpu(), cpool0)
    finally:
        kda.kda_testing_set_first_wait_tries(-1)
    d2 = dict(d, pool=pool0.clone(), conv_pool=cpool0.clone())
    out, pool, ck, offs, status, cpool = run_prefill_conv(kda, d2, w, DEV)
    assert int(status.item()) == 0
    o_ref, p_ref, ck_ref, offs_ref, c_ref = oracle_prefill_conv(oracle, d2, w)
    tol = tol_for(w.state_dtype)
    assert excess_error(out, o_ref) <= tol
    touched = d["state_indices"].long().tolist()
    assert max_abs(pool[touched], p_ref[touched]) <= tol
    cpool_cpu = cpool.cpu()
    for s_ in touched:
        assert torch.equal(cpool_cpu[s_].double(), torch.as_tensor(c_ref[s_]).double()), s_
    assert offs.cpu().tolist() == offs_ref.tolist()
