"""The seeded input recipe: shapes, dtypes and value ranges per workload."""
import numpy as np
import torch

import kda_inputs as KI


def test_tiny_workload_recipe():
    d = KI.make_inputs(KI.WORKLOADS["tiny_T64_H1"])
    assert d["q"].dtype == torch.bfloat16 and d["q"].shape == (64, 1, 128)
    assert d["v"].dtype == torch.bfloat16 and d["g"].dtype == torch.float32
    assert d["beta"].shape == (64, 1) and d["initial_state"] is None
    nq = torch.linalg.vector_norm(d["q"].float(), dim=-1)
    nk = torch.linalg.vector_norm(d["k"].float(), dim=-1)
    assert torch.allclose(nq, torch.ones_like(nq), atol=1e-2)
    assert torch.allclose(nk, torch.ones_like(nk), atol=1e-2)
    assert (d["g"] <= 0).all() and (d["beta"] > 0).all() and (d["beta"] < 1).all()
    assert d["cu_seqlens"].tolist() == [0, 64]


def test_seeded_and_deterministic():
    a = KI.make_inputs(KI.WORKLOADS["tiny_T64_H1"])
    b = KI.make_inputs(KI.WORKLOADS["tiny_T64_H1"])
    for key in ("q", "k", "v", "g", "beta"):
        assert torch.equal(a[key], b[key])


def test_varlen_lengths():
    gen = torch.Generator().manual_seed(3)
    lens = KI.draw_varlen_lengths(gen, 8192, 16)
    assert len(lens) == 16 and sum(lens) == 8192
    assert min(lens) >= 64 and all(L % 16 for L in lens)


def test_varlen_workload_cu_seqlens():
    w = KI.WORKLOADS["varlen16_T8192_H64"]
    small = KI.Workload("v", seed=w.seed, T=2048, H=2, n_seqs=16, varlen=True, init_state=True)
    d = KI.make_inputs(small)
    cu = d["cu_seqlens"].numpy()
    assert cu[0] == 0 and cu[-1] == 2048 and np.all(np.diff(cu) >= 64)
    assert d["initial_state"].shape == (16, 2, 128, 128)
    assert abs(float(d["initial_state"].std()) - 0.02) < 2e-3


def test_make_case_zero_lengths():
    d = KI.make_case([3, 0, 17], H=2, seed=5, init_state=True)
    assert d["cu_seqlens"].tolist() == [0, 3, 3, 20]
    assert d["q"].shape == (20, 2, 128)
