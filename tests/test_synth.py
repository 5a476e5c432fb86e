"""The seeded input generator: bf16 rounding, determinism, shapes and the documented
distributions (x ~ N(0,1); B, C ~ N(0, 1/(N R)); dt = softplus(N(-2, 0.5));
A = -exp(U(0, ln 16)); lambda = sigmoid(N(0, 1)); theta ~ N(0, 1))."""
import numpy as np
import pytest
import torch

from state_space_sequence_trapezoidal_b300 import synth


def test_round_bf16_matches_torch_round_to_nearest_even():
    rng = np.random.Generator(np.random.PCG64(0))
    a = np.concatenate([
        rng.standard_normal(100000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 100000),
        # exact ties between two bf16 values (lower 16 bits 0x8000), both parities
        (np.arange(1, 2000, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
        np.array([0.0, -0.0, 1e-40, -1e-40, 3.0e38, -3.0e38, np.inf, -np.inf], np.float32),
    ]).astype(np.float32)
    ours = synth.round_bf16(a)
    ref = torch.from_numpy(a).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(ours.view(np.uint32), ref.view(np.uint32))


def test_inputs_are_deterministic_and_shaped_like_the_layouts():
    a = synth.make_inputs(2, 5, 3, 8, 6, 2, 123, "bf16")
    b = synth.make_inputs(2, 5, 3, 8, 6, 2, 123, "bf16")
    c = synth.make_inputs(2, 5, 3, 8, 6, 2, 124, "bf16")
    shapes = {"x": (2, 5, 3, 2, 8), "B": (2, 5, 3, 2, 6), "C": (2, 5, 3, 2, 6), "dt": (2, 5, 3),
              "lambda": (2, 5, 3), "theta": (2, 5, 3, 3), "A": (3,)}
    for k, shp in shapes.items():
        assert a[k].shape == shp and a[k].dtype == np.float32, k
        np.testing.assert_array_equal(a[k], b[k])
        assert not np.array_equal(a[k], c[k]), k
    # bf16 workloads are bf16-exact (A stays float32)
    for k in ("x", "B", "C", "dt", "lambda", "theta"):
        np.testing.assert_array_equal(a[k], synth.round_bf16(a[k]))


def test_a_seed_keeps_a_fixed_across_decode_steps():
    s0 = synth.make_inputs(1, 1, 4, 8, 4, 1, synth.decode_step_seed(7, 0), "bf16", A_seed=7)
    s1 = synth.make_inputs(1, 1, 4, 8, 4, 1, synth.decode_step_seed(7, 1), "bf16", A_seed=7)
    np.testing.assert_array_equal(s0["A"], s1["A"])
    assert not np.array_equal(s0["x"], s1["x"])


@pytest.mark.parametrize("N,R", [(128, 1), (64, 4)])
def test_distributions(N, R):
    d = synth.make_inputs(4, 512, 8, 64, N, R, 99, "f32")
    assert abs(d["x"].mean()) < 0.01 and abs(d["x"].std() - 1.0) < 0.01
    sd = 1.0 / np.sqrt(N * R)
    assert abs(d["B"].std() / sd - 1.0) < 0.01 and abs(d["C"].std() / sd - 1.0) < 0.01
    z = np.log(np.expm1(d["dt"].astype(np.float64)))          # inverse softplus
    assert abs(z.mean() + 2.0) < 0.02 and abs(z.std() - 0.5) < 0.02
    assert np.all(d["dt"] > 0)
    lam = d["lambda"].astype(np.float64)
    assert np.all((lam > 0) & (lam < 1))
    logit = np.log(lam / (1 - lam))
    assert abs(logit.mean()) < 0.02 and abs(logit.std() - 1.0) < 0.02
    assert abs(d["theta"].std() - 1.0) < 0.01
    assert np.all((d["A"] <= -1.0) & (d["A"] >= -16.0))


def test_workloads_are_the_benchmark_shapes():
    w = synth.WORKLOADS["siso-prefill-bf16-b8-t4096-h32-p64-n128"]
    assert (w.B, w.T, w.H, w.P, w.N, w.R, w.dtype) == (8, 4096, 32, 64, 128, 1, "bf16")
    w = synth.WORKLOADS["mimo-r4-decode-bf16-b256-h32-p64-n64"]
    assert (w.B, w.H, w.P, w.N, w.R, w.decode_steps) == (256, 32, 64, 64, 4, 1000)
    assert len({w.name for w in synth.WORKLOADS.values()}) == 6
