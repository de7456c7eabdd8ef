"""The seeded input generators: determinism, rounding and distributions."""
import numpy as np
import torch

import synth


def test_deterministic_and_stream_independent():
    a = synth.normal(5, 1, 1000)
    b = synth.normal(5, 1, 1000)
    c = synth.normal(5, 2, 1000)
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    # a prefix does not depend on how many values are drawn
    assert np.array_equal(synth.normal(5, 1, 10), a[:10])
    assert abs(a.mean()) < 0.15 and abs(a.std() - 1) < 0.1


def test_bf16_rounding_matches_torch_rne():
    x = synth.normal(0, 3, 100000) * 3.0
    ours = synth.round_to(x, "bf16")
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(ours, ref)


def test_workload_shapes_and_ranges():
    d = synth.qdelta_inputs(2, 70, 3, 16, 8, seed=1)
    assert d["q"].shape == (2, 70, 3, 16) and d["v"].shape == (2, 70, 3, 8)
    assert d["alpha"].shape == (2, 70, 3) and d["S0"] is None
    assert np.all((d["beta"] > 0) & (d["beta"] < 1))
    assert np.all((d["alpha"] > 0.9) & (d["alpha"] <= 1))
    assert np.allclose(np.linalg.norm(d["q"], axis=-1), 1, atol=1e-2)
    g = synth.qdelta_inputs(1, 8, 1, 8, 8, seed=1, mode="deltanet")
    assert g["alpha"] is None and g["lam"] is None
    e = synth.qed_inputs(1, 9, 2, 8, 4, seed=3)
    assert e["g"].shape == (1, 9, 2, 8) and e["w"].shape == (1, 9, 2, 4) and e["lam_h"].shape == (2,)
    assert np.all(e["g"] < 0)


def test_mean_alpha_bisection():
    mu = synth.alpha_mu_for_mean(0.995)
    z = synth.normal(9, 9, 200000, mean=mu, std=0.5)
    assert abs(np.mean(np.exp(-np.logaddexp(0, z))) - 0.995) < 2e-4
    assert -5.6 < mu < -5.2


def test_backward_prologue_and_eda_generators():
    """The cotangent, projection and EDA generators: seeded, of the stated shapes and
    distributions, and independent of each other's streams."""
    c1 = synth.cotangents(2, 10, 3, 16, 8, seed=5, dtype="bf16")
    c2 = synth.cotangents(2, 10, 3, 16, 8, seed=5, dtype="bf16")
    assert c1["dO"].shape == (2, 10, 3, 8) and c1["dS_final"].shape == (2, 3, 8, 16)
    assert np.array_equal(c1["dO"], c2["dO"]) and np.array_equal(c1["dS_final"], c2["dS_final"])
    assert synth.cotangents(1, 4, 1, 16, 16, seed=5, final_state=False)["dS_final"] is None
    big = synth.cotangents(1, 512, 4, 64, 64, seed=6, dtype="f32")
    assert abs(big["dO"].mean()) < 0.02 and abs(big["dO"].std() - 1.0) < 0.02

    r = synth.qdelta_raw_inputs(1, 256, 4, 64, 64, seed=7, dtype="f32")
    assert abs(np.linalg.norm(r["q"], axis=-1).mean() - 8.0) < 0.5           # raw: |q| ~ sqrt(64)
    assert abs(r["alpha"].mean() + 4.0) < 0.05 and abs(r["alpha"].std() - 0.5) < 0.05
    assert abs(r["beta"].mean()) < 0.1 and abs(r["beta"].std() - 1.0) < 0.1

    e = synth.eda_inputs(1, 64, 2, 32, 32, seed=8, dtype="f32")
    np.testing.assert_allclose(np.linalg.norm(e["e"], axis=-1), 1.0, atol=1e-6)
    assert not np.allclose(e["e"], e["q"])
    eq = synth.eda_inputs(1, 64, 2, 32, 32, seed=8, dtype="f32", erase="query", beta=False)
    assert np.array_equal(eq["e"], eq["q"]) and eq["beta"] is None
