"""Shapes and structure of the seeded synthetic workloads (CPU only)."""
import numpy as np
import torch

import oracle
import workloads as W


def test_sched_lengths_composition():
    lens = W.SCHED.seqlens
    assert len(lens) == 8 and sum(lens) == 4096 and min(lens) >= 64
    assert W.sched_lengths(4096, 8, 64, 2) == lens  # seeded, reproducible


def test_varlen_checkpoint_count():
    d = W.make_prefill(W.VARLEN)
    offs = oracle.checkpoint_offsets(d["cu_seqlens"], W.VARLEN.checkpoint_every)
    assert offs.tolist() == [0, 0, 2, 5, 13]
    assert d["q"].dtype == torch.bfloat16 and d["pool"].dtype == torch.float32
    assert len(set(d["state_indices"].tolist())) == 4


def test_sched_slots_in_top_half():
    d = W.make_prefill(W.SCHED.replace(num_slots=512, H=2))
    idx = d["state_indices"].numpy()
    assert np.all((idx >= 256) & (idx < 512)) and len(set(idx.tolist())) == 8


def test_input_distributions():
    d = W.make_prefill(W.TINY)
    q = d["q"].double()
    assert torch.allclose(q.norm(dim=-1), torch.ones(64, 2, dtype=torch.float64), atol=1e-6)
    assert torch.all(d["g"] < 0) and torch.all((d["beta"] > 0) & (d["beta"] < 1))
    assert torch.all(d["pool"] == 0)
