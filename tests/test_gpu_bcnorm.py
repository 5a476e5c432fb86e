"""GPU parity of the fused BCNorm + bias prologue (m3_ssm_prefill_bcnorm and
m3_ssm_decode_step_bcnorm, paper section 3.4) through the C ABI against the oracle chain
oracle.bcnorm (RMS normalisation, weight, per-head bias) -> oracle.scan (the recurrence).

Raw B, C rows carry random scales, so a kernel that skipped or misplaced the normalisation
fails.  The state keeps the raw previous B, which both sides normalise when folding the
previous token's trapezoid term; the exit state's prev_B must be the raw last B, bit for bit.
Tolerances as in the other parity tests: max|gpu - oracle| / RMS <= 2e-2 (bf16 inputs) or
1e-4 (fp32 inputs)."""
import numpy as np
import pytest
import torch

import oracle
import state_space_sequence_trapezoidal_b300 as m3
from oracle.bcnorm import bc_prologue_layout
from state_space_sequence_trapezoidal_b300 import synth
from tests import parity as P

pytestmark = pytest.mark.gpu


def norm_to_device(prm: dict, dtype: str, drop=()):
    t = P.tdtype(dtype)
    return m3.BCNorm(**{k: (None if k in drop else torch.from_numpy(prm[k]).to("cuda", t))
                        for k in ("B_weight", "B_bias", "C_weight", "C_bias")}, eps=prm["eps"])


def normed(prm: dict, drop=()):
    """The oracle's view of the parameters (ones / zeros where the GPU gets None)."""
    q = dict(prm)
    for k in drop:
        q[k] = np.ones_like(prm[k]) if k.endswith("weight") else np.zeros_like(prm[k])
    return q


def oracle_bcnorm(raw: dict, prm: dict, slices, state_raw: dict | None = None):
    """oracle.bcnorm then oracle.scan on the chosen (b, h) sequences; returns y and the exit
    state with prev_B replaced by the raw last B (what the library stores)."""
    lay = dict(raw)
    lay["B"] = bc_prologue_layout(raw["B"], prm["B_weight"], prm["B_bias"], prm["eps"])
    lay["C"] = bc_prologue_layout(raw["C"], prm["C_weight"], prm["C_bias"], prm["eps"])
    st = None
    if state_raw is not None:
        st = dict(state_raw)
        st["prev_B"] = bc_prologue_layout(state_raw["prev_B"][:, None], prm["B_weight"],
                                          prm["B_bias"], prm["eps"])[:, 0]
    y, sr = P.run_oracle(lay, slices, st)
    T = raw["x"].shape[1]
    if T > 0:
        sr["prev_B"] = P.pick(raw["B"][:, T - 1], slices, False)
    return y, sr


def raw_prior_state(B, H, N, Pd, R, dtype, prm, seed, T0=96):
    """The exit state of 96 seeded raw tokens through the oracle chain (raw prev_B)."""
    raw = synth.make_raw_bc(synth.make_inputs(B, T0, H, Pd, N, R, seed, dtype), seed + 1, dtype)
    sl = P.all_slices(B, H)
    _, sr = oracle_bcnorm(raw, prm, sl)
    out = {k: np.zeros((B, H) + v.shape[1:], np.float32) for k, v in sr.items()}
    for i, (b, h) in enumerate(sl):
        for k in sr:
            out[k][b, h] = sr[k][i]
    return out


def run_prefill(raw_dev, norm, h0=None, out_dtype=torch.float32):
    x = raw_dev["x"]
    Bsz, T, H, R, Pd = x.shape
    N = raw_dev["B"].shape[-1]
    hT = m3.State.zeros(Bsz, H, N, Pd, R, dtype=x.dtype)
    ws = m3.prefill_workspace(x, raw_dev["dt"], raw_dev["theta"], out_dtype)
    y = m3.m3_ssm_prefill_bcnorm(x, raw_dev["B"], raw_dev["C"], raw_dev["dt"], raw_dev["A"],
                                 raw_dev["lambda"], raw_dev["theta"], norm, h0, hT=hT,
                                 workspace=ws, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert m3.m3_ssm_device_status(ws) == m3.M3_OK
    return y, hT


def check(y, hT, yr, sr, sl, dtype):
    e = P.rel_err(P.pick(y.float().cpu().numpy(), sl, True), yr)
    assert e <= P.TOL[dtype], e
    P.check_state({k: P.pick(v, sl, False) for k, v in P.state_to_host(hT).items()}, sr, dtype)


@pytest.mark.parametrize("N,R", [(128, 1), (64, 4), (128, 2), (64, 8), (64, 1), (128, 4)])
@pytest.mark.parametrize("fresh", [False, True])
def test_bcnorm_tensor_core_prefill(N, R, fresh):
    """Three chunks and a ragged tail; with and without an entry state (raw prev_B folded)."""
    B, H, Pd = 2, 3, 64
    T = 3 * (128 // R) + (128 // R) // 2 + 3
    prm = synth.make_bcnorm_params(N, H, R, 50 + N + R)
    raw = synth.make_raw_bc(synth.make_inputs(B, T, H, Pd, N, R, 5000 + N + R, "bf16"), 7)
    st0 = None if fresh else raw_prior_state(B, H, N, Pd, R, "bf16", prm, 9)
    y, hT = run_prefill(P.to_device(raw, "bf16"), norm_to_device(prm, "bf16"),
                        None if fresh else P.state_to_device(st0, "bf16"))
    sl = P.all_slices(B, H)
    yr, sr = oracle_bcnorm(raw, prm, sl, st0)
    check(y, hT, yr, sr, sl, "bf16")


@pytest.mark.parametrize("N,R,T", [(128, 1, 1500), (64, 4, 600)])
def test_bcnorm_segmented_long_sequence(N, R, T):
    """Few (batch row, head) pairs: the first pass (B only) and the scan's fold use the norm."""
    B, H, Pd = 1, 4, 64
    prm = synth.make_bcnorm_params(N, H, R, 60 + N + R)
    raw = synth.make_raw_bc(synth.make_inputs(B, T, H, Pd, N, R, 5100 + N + T, "bf16"), 8)
    d = P.to_device(raw, "bf16")
    assert m3.prefill_workspace(d["x"], d["dt"], d["theta"]).numel() > 256
    st0 = raw_prior_state(B, H, N, Pd, R, "bf16", prm, 10)
    y, hT = run_prefill(d, norm_to_device(prm, "bf16"), P.state_to_device(st0, "bf16"))
    sl = P.all_slices(B, H)
    yr, sr = oracle_bcnorm(raw, prm, sl, st0)
    check(y, hT, yr, sr, sl, "bf16")


@pytest.mark.parametrize("drop", [("B_weight", "C_weight", "B_bias", "C_bias"), ("B_bias",),
                                  ("C_weight",)])
def test_bcnorm_absent_parameters_are_ones_and_zeros(drop):
    B, H, Pd, N, R, T = 2, 2, 64, 128, 1, 300
    prm = synth.make_bcnorm_params(N, H, R, 70)
    raw = synth.make_raw_bc(synth.make_inputs(B, T, H, Pd, N, R, 5200, "bf16"), 11)
    st0 = raw_prior_state(B, H, N, Pd, R, "bf16", normed(prm, drop), 12)
    y, hT = run_prefill(P.to_device(raw, "bf16"), norm_to_device(prm, "bf16", drop),
                        P.state_to_device(st0, "bf16"))
    sl = P.all_slices(B, H)
    yr, sr = oracle_bcnorm(raw, normed(prm, drop), sl, st0)
    check(y, hT, yr, sr, sl, "bf16")


@pytest.mark.parametrize("N,Pd,R,T", [(16, 16, 1, 70), (6, 8, 2, 37), (32, 12, 4, 41)])
def test_bcnorm_fp32_recurrent_prefill(N, Pd, R, T):
    B, H = 2, 3
    prm = synth.make_bcnorm_params(N, H, R, 80 + N, "f32")
    raw = synth.make_raw_bc(synth.make_inputs(B, T, H, Pd, N, R, 5300 + N, "f32"), 13, "f32")
    st0 = raw_prior_state(B, H, N, Pd, R, "f32", prm, 14)
    y, hT = run_prefill(P.to_device(raw, "f32"), norm_to_device(prm, "f32"),
                        P.state_to_device(st0, "f32"))
    sl = P.all_slices(B, H)
    yr, sr = oracle_bcnorm(raw, prm, sl, st0)
    check(y, hT, yr, sr, sl, "f32")


@pytest.mark.parametrize("N,Pd,R,dtype", [(128, 64, 1, "bf16"), (64, 64, 4, "bf16"),
                                          (16, 16, 1, "f32"), (6, 8, 2, "f32"),
                                          (32, 12, 8, "bf16")])
def test_bcnorm_decode_steps(N, Pd, R, dtype):
    B, H, K = 3, 5, 6
    prm = synth.make_bcnorm_params(N, H, R, 90 + N + R, dtype)
    st0 = raw_prior_state(B, H, N, Pd, R, dtype, prm, 15)
    state = P.state_to_device(st0, dtype)
    norm = norm_to_device(prm, dtype)
    sl = P.all_slices(B, H)
    ref = {k: v.copy() for k, v in st0.items()}
    for s in range(K):
        one = synth.make_inputs(B, 1, H, Pd, N, R, synth.decode_step_seed(600, s), dtype,
                                A_seed=600)
        raw = synth.make_raw_bc(one, 700 + s, dtype)
        dev = P.to_device({k: (v[:, 0] if k != "A" else v) for k, v in raw.items()}, dtype)
        y = m3.m3_ssm_decode_step_bcnorm(state, dev["x"], dev["B"], dev["C"], dev["dt"], dev["A"],
                                         dev["lambda"], dev["theta"], norm)
        torch.cuda.synchronize()
        yr, sr = oracle_bcnorm(raw, prm, sl, ref)
        e = P.rel_err(P.pick(y.cpu().numpy(), sl, False), yr[:, 0])
        assert e <= P.TOL[dtype], (s, e)
        ref = {k: _unpick(v, sl, B, H) for k, v in sr.items()}
    P.check_state({k: P.pick(v, sl, False) for k, v in P.state_to_host(state).items()},
                  {k: P.pick(v, sl, False) for k, v in ref.items()}, dtype)


def _unpick(stack, slices, B, H):
    out = np.zeros((B, H) + stack.shape[1:], stack.dtype)
    for i, (b, h) in enumerate(slices):
        out[b, h] = stack[i]
    return out


@pytest.mark.parametrize("N,R", [(128, 1), (64, 4)])
def test_bcnorm_prefill_then_decode(N, R):
    """A fused prefill hands its state (raw prev_B) to fused decode steps: all against the
    oracle run over the whole sequence."""
    B, H, Pd, T, K = 2, 3, 64, 300, 24
    prm = synth.make_bcnorm_params(N, H, R, 95)
    raw = synth.make_raw_bc(synth.make_inputs(B, T + K, H, Pd, N, R, 5400 + N, "bf16"), 16)
    pre = {k: (v[:, :T] if k != "A" else v) for k, v in raw.items()}
    d = P.to_device(raw, "bf16")
    norm = norm_to_device(prm, "bf16")
    y, st = run_prefill(P.to_device(pre, "bf16"), norm)
    ys = [m3.m3_ssm_decode_step_bcnorm(st, d["x"][:, t].contiguous(), d["B"][:, t].contiguous(),
                                       d["C"][:, t].contiguous(), d["dt"][:, t].contiguous(),
                                       d["A"], d["lambda"][:, t].contiguous(),
                                       d["theta"][:, t].contiguous(), norm)
          for t in range(T, T + K)]
    torch.cuda.synchronize()
    got = np.concatenate([y.cpu().numpy(), torch.stack(ys, 1).cpu().numpy()], axis=1)
    sl = P.all_slices(B, H)
    yr, sr = oracle_bcnorm(raw, prm, sl)
    assert P.rel_err(P.pick(got, sl, True), yr) <= P.TOL["bf16"]
    P.check_state({k: P.pick(v, sl, False) for k, v in P.state_to_host(st).items()}, sr, "bf16")


def test_bcnorm_full_size_headline_sampled():
    """The headline shape (B8 T4096 H32 P64 N128) through the fused prologue, 8 sampled
    sequences against the oracle chain."""
    w = synth.WORKLOADS["siso-prefill-bf16-b8-t4096-h32-p64-n128"]
    prm = synth.make_bcnorm_params(w.N, w.H, w.R, 99)
    raw = synth.make_raw_bc(synth.make_inputs(w.B, w.T, w.H, w.P, w.N, w.R, w.seed, w.dtype), 17)
    y, hT = run_prefill(P.to_device(raw, "bf16"), norm_to_device(prm, "bf16"))
    sl = P.sample_slices(w.B, w.H, 8, w.seed)
    yr, sr = oracle_bcnorm(raw, prm, sl)
    check(y, hT, yr, sr, sl, "bf16")
