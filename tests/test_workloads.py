"""CPU tests of the seeded input generators (shapes, determinism, recipe)."""
import numpy as np
import torch

import workloads


def test_shapes_dtypes_and_determinism():
    w = workloads.TINY
    a = workloads.make_inputs(w, 5, "cpu")
    b = workloads.make_inputs(w, 5, "cpu")
    c = workloads.make_inputs(w, 6, "cpu")
    assert a["zt"].shape == (4, 5, 1024) and a["zt"].dtype == torch.float32
    assert a["zd"].shape == (4, 4, 1024)
    assert a["x"].shape == (4, 4) and a["x"].dtype == torch.int32
    assert a["u"].shape == (4, 5)
    for k in a:
        assert torch.equal(a[k], b[k])
    assert not torch.equal(a["zt"], c["zt"])
    assert ((a["u"] >= 0) & (a["u"] < 1)).all()
    assert ((a["x"] >= 0) & (a["x"] < 1024)).all()


def test_bf16_recipe_and_spikes():
    w = workloads.LLAMA3_VOCAB.scaled(B=2, V=4096)
    a = workloads.make_inputs(w, 1, "cpu")
    assert a["zt"].dtype == torch.bfloat16
    zt = a["zt"].float()
    # one +12 spike per row: the row max sits well above the N(0, 2.5^2) bulk
    assert (zt.amax(-1) > 8).float().mean() > 0.9
    bulk = zt.flatten()
    assert abs(bulk.std().item() - 2.5) < 0.1
    noise = (a["zd"].float() - zt[:, :w.K]).flatten()
    assert abs(noise.std().item() - 0.8) < 0.05


def test_fly_halves_and_greedy_drafts():
    w = workloads.FLY.scaled(B=4, V=4096)
    a = workloads.make_inputs(w, 2, "cpu")
    zt = a["zt"].float()
    assert zt[:2].std() < 0.6 and zt[2:].std() > 3.0
    assert torch.equal(a["x"], a["zd"].float().argmax(-1).to(torch.int32))


def test_temperature_recipe():
    w = workloads.ESTIMATOR.scaled(B=8, V=2048)
    a = workloads.make_inputs(w, 3, "cpu")
    s = a["zt"].float().std(-1)
    # N(0, 3^2) / T with T ~ U(0.5, 2): row std between 1.5 and 6
    assert s.min() > 1.3 and s.max() < 6.5


def test_numpy_view_of_bf16_is_raw_bits():
    z = torch.tensor([1.0, -2.5, 3.0], dtype=torch.bfloat16)
    n = workloads.to_numpy_logits(z)
    assert n.dtype == np.uint16
    back = (n.astype(np.uint32) << 16).view(np.float32)
    np.testing.assert_array_equal(back, [1.0, -2.5, 3.0])
