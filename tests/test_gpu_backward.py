"""GPU parity of the prefill's backward pass (m3_ssm_prefill_backward) against the gradient
oracle (oracle/grad.py, pinned by finite differences of the C oracle).

Every gradient tensor -- dx, dB, dC, ddt, dlambda, dtheta, dA, dh0 -- is compared element by
element: max|gpu - oracle| / rms(oracle) <= 1e-4.  The kernel computes in fp32 from the exact
input values (bf16 inputs are upcast exactly), so the fp32 tolerance applies to both input
dtypes.  Shapes span the kernels' chunk lengths (32, 16 and 4 tokens; 8 to 64 (token, rank)
rows), chunk boundaries inside and at the end of the sequence, ragged last chunks, a single
token, and the entry-state fold.
"""
import numpy as np
import pytest
import torch

import state_space_sequence_trapezoidal_b300 as m3
from oracle import grad as OG
import oracle
from state_space_sequence_trapezoidal_b300 import synth
from tests import parity as P

pytestmark = pytest.mark.gpu

TOL = 1e-4
KEYS = {"dx": "x", "dB": "Bm", "dC": "Cm", "ddt": "dt", "dlambda": "lam", "dtheta": "theta"}


def run(B, T, H, Pd, N, R, dtype, seed, with_state, dy_dtype=torch.float32, slices=None):
    inp = synth.make_inputs(B, T, H, Pd, N, R, seed, dtype)
    rng = np.random.Generator(np.random.PCG64(seed + 1))
    dy = rng.standard_normal((B, T, H, R, Pd)).astype(np.float32)
    if dy_dtype == torch.bfloat16:
        dy = synth.round_bf16(dy)
    dhT = rng.standard_normal((B, H, N, Pd)).astype(np.float32) * 0.1
    st0 = P.prior_state(B, H, N, Pd, R, dtype, seed + 2) if with_state else None
    d = P.to_device(inp, dtype)
    h0 = P.state_to_device(st0, dtype) if with_state else None
    g = m3.m3_ssm_prefill_backward(d["x"], d["B"], d["C"], d["dt"], d["A"], d["lambda"], d["theta"],
                                   torch.from_numpy(dy).to("cuda", dy_dtype), h0,
                                   dhT=torch.from_numpy(dhT).cuda(), want_dh0=True)
    torch.cuda.synchronize()
    sl = slices or P.all_slices(B, H)
    layout = dict(inp)
    if st0 is not None:
        layout["state"] = st0
    o = oracle.gather(layout, sl)
    dys = np.stack([dy[b, :, h] for b, h in sl])
    dhs = np.stack([dhT[b, h] for b, h in sl])
    ref = OG.grads(o["x"], o["Bm"], o["Cm"], o["dt"], o["A"], o["lam"], o["theta"], dys, dhs,
                   o.get("state"))
    return g, ref, sl


def check(g, ref, sl, H, full_batch):
    for k, rk in KEYS.items():
        got = P.pick(g[k].cpu().numpy(), sl, True)
        e = P.rel_err(got, ref[rk])
        assert e <= TOL, (k, e)
    e = P.rel_err(P.pick(g["dh0"].cpu().numpy(), sl, False), ref["h0"])
    assert e <= TOL, ("dh0", e)
    if full_batch:  # dA[h] sums over every batch row
        want = np.zeros(H)
        for (b, h), v in zip(sl, ref["A"]):
            want[h] += v
        got = g["dA"].cpu().numpy()
        assert np.max(np.abs(got - want)) <= TOL * np.sqrt(np.mean(want ** 2)) * 10, (got, want)


@pytest.mark.parametrize("N,Pd,R,T", [(16, 16, 1, 40), (8, 12, 2, 37), (32, 32, 4, 20),
                                      (128, 64, 1, 50), (64, 64, 4, 33), (128, 64, 8, 9),
                                      (6, 4, 1, 1), (128, 64, 1, 130), (64, 64, 4, 70),
                                      (128, 64, 2, 100), (16, 8, 1, 64)])
@pytest.mark.parametrize("with_state", [False, True])
def test_backward_f32_matches_gradient_oracle(N, Pd, R, T, with_state):
    B, H = 2, 2
    g, ref, sl = run(B, T, H, Pd, N, R, "f32", 100 + N + Pd + R + T, with_state)
    check(g, ref, sl, H, True)


@pytest.mark.parametrize("N,R", [(128, 1), (64, 4)])
def test_backward_bf16_inputs_and_bf16_dy(N, R):
    B, H, Pd, T = 2, 3, 64, 45
    g, ref, sl = run(B, T, H, Pd, N, R, "bf16", 300 + N + R, True, dy_dtype=torch.bfloat16)
    check(g, ref, sl, H, True)


def test_backward_rerun_is_bit_identical():
    B, H, Pd, N, R, T = 2, 2, 64, 128, 1, 40
    inp = synth.make_inputs(B, T, H, Pd, N, R, 7, "bf16")
    d = P.to_device(inp, "bf16")
    dy = torch.randn(B, T, H, R, Pd, device="cuda")
    a = m3.m3_ssm_prefill_backward(d["x"], d["B"], d["C"], d["dt"], d["A"], d["lambda"], d["theta"], dy)
    b = m3.m3_ssm_prefill_backward(d["x"], d["B"], d["C"], d["dt"], d["A"], d["lambda"], d["theta"], dy)
    torch.cuda.synchronize()
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_backward_full_size_sampled():
    """The benchmark's backward workload (the headline prefill shape, B8 T4096 H32 N128) in the
    benchmark's launch configuration; sampled (b, h) sequences against the oracle."""
    w = synth.WORKLOADS["siso-prefill-bf16-b8-t4096-h32-p64-n128"]
    sl = P.sample_slices(w.B, w.H, 2, 53)
    g, ref, sl = run(w.B, w.T, w.H, w.P, w.N, w.R, "bf16", w.seed, False, slices=sl)
    check(g, ref, sl, w.H, False)


def test_backward_mimo_full_size_sampled():
    """The MIMO rank-4 prefill shape (B8 T4096 H32 N64, 16-token chunks: 256 chunk scans per
    sequence) through its compile-time-specialised kernels; sampled (b, h) sequences against the
    oracle, with an entry state."""
    w = synth.WORKLOADS["mimo-r4-prefill-bf16-b8-t4096-h32-p64-n64"]
    sl = P.sample_slices(w.B, w.H, 2, 71)
    g, ref, sl = run(w.B, w.T, w.H, w.P, w.N, w.R, "bf16", w.seed, True, slices=sl)
    check(g, ref, sl, w.H, False)
