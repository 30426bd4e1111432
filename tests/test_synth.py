"""The seeded input generator: shapes, determinism and workload structure."""
import torch

from synth import WORKLOAD_ORDER, make_inputs, varlen_lengths, workload


def test_deterministic_and_shapes():
    w = workload(0)
    a, b = make_inputs(w), make_inputs(w)
    for key in ("q", "k", "v", "g", "beta", "h0", "do", "dht"):
        assert torch.equal(a[key], b[key]), key
    assert a["q"].shape == (1, 256, 2, 64) and a["v"].shape == (1, 256, 2, 64)
    assert a["h0"].shape == (1, 2, 64, 64)
    assert torch.allclose(a["q"].float().norm(dim=-1), torch.ones(1, 256, 2), atol=1e-5)
    assert (a["g"] <= 0).all() and ((a["beta"] > 0) & (a["beta"] < 1)).all()


def test_varlen_lengths():
    lens = varlen_lengths(8, 32768, 512, 8192, 2)
    assert len(lens) == 8 and sum(lens) == 32768
    assert all(512 <= x <= 8192 for x in lens)


def test_zero_gate_heads():
    w = workload("train_b2_t8192_h64").scaled(T=64)
    x = make_inputs(w)
    zero = (x["g"] == 0).all(dim=1).all(dim=0)
    assert int(zero.sum()) == 6


def test_workload_table():
    assert len(WORKLOAD_ORDER) == 5
    assert workload(1).Hv // workload(1).Hq == 2 and workload(4).Hv // workload(4).Hq == 4
    assert workload(3).B * workload(3).Hv == 8
