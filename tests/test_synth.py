"""The seeded input generator: shapes, dtypes, determinism, disjoint flags."""
import numpy as np
import torch

from first_order_linear_gb300 import synth


def test_value_rollout_shapes_and_determinism():
    a = synth.value_rollout(8, 16, seed=0)
    b = synth.value_rollout(8, 16, seed=0)
    for k in a:
        assert torch.equal(a[k], b[k])
    assert a["rewards"].shape == (8, 16) and a["rewards"].dtype == torch.float32
    assert a["bootstrap"].shape == (8,)
    assert a["terminated"].dtype == torch.uint8
    assert not torch.any(a["terminated"] & a["truncated"])


def test_no_trunc_keeps_other_draws():
    a = synth.value_rollout(64, 32, seed=3, with_trunc=True)
    b = synth.value_rollout(64, 32, seed=3, with_trunc=False)
    assert b["truncated"] is None and b["trunc_value"] is None
    assert torch.equal(a["rewards"], b["rewards"])
    assert torch.equal(a["terminated"], b["terminated"])


def test_policy_rollouts():
    v = synth.vtrace_rollout(16, 8, seed=1)
    assert v["logp_target"].shape == (16, 8)
    assert torch.all(v["logp_target"] <= 0) and torch.all(v["logp_behaviour"] <= 0)
    r = synth.retrace_rollout(4, 8, seed=2)
    assert r["q"].shape == (4, 8, 18) and r["pi"].shape == (4, 8, 18)
    assert torch.allclose(r["pi"].sum(-1), torch.ones(4, 8), atol=1e-5)
    assert r["actions"].dtype == torch.int32 and int(r["actions"].max()) < 18
    assert torch.all(r["mu_a"] > 0)


def test_numpy_and_time_major_roundtrip():
    d = synth.numpy(synth.forward_rollout(4, 6, seed=5))
    assert isinstance(d["x_f32"], np.ndarray) and d["x_i32"].dtype == np.int32
    x = np.arange(24, dtype=np.float32).reshape(4, 6)
    tm = synth.to_time_major(x)
    assert tm.shape == (6, 4) and tm.flags.c_contiguous
    assert np.array_equal(synth.from_time_major(tm), x)
    q = torch.arange(48, dtype=torch.float32).reshape(2, 4, 6)
    assert torch.equal(synth.from_time_major(synth.to_time_major(q)), q)
