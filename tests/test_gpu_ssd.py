"""GPU parity of the Mamba-2 special case (m3_ssd_prefill / m3_ssd_decode_step) against the
fp64 oracle run with lambda = 1 and theta = 0.

That reading of the oracle is pinned on its own in test_oracle_pins (the exponential-Euler
loop of Eq. (4)); here the specialised kernels, with the rotation and the lambda terms
compiled out, must reproduce it within the same tolerances as the full method.
"""
import numpy as np
import pytest
import torch

import state_space_sequence_trapezoidal_b300 as m3
from state_space_sequence_trapezoidal_b300 import synth
from tests import parity as P

pytestmark = pytest.mark.gpu


def ssd_inputs(B, T, H, Pd, N, seed, dtype):
    """Seeded inputs with lambda = 1 and theta = 0 (what the special case computes)."""
    inp = synth.make_inputs(B, T, H, Pd, N, 1, seed, dtype)
    inp["lambda"] = np.ones_like(inp["lambda"])
    inp["theta"] = np.zeros_like(inp["theta"])
    return inp


def ssd_state(h: np.ndarray, N: int, Pd: int) -> dict:
    """Oracle state for an SSD entry state h: no angle, no previous token (its weight
    (1 - lambda) dt vanishes anyway)."""
    B, H = h.shape[:2]
    return {"h": h, "phi": np.zeros((B, H, N // 2), np.float32),
            "prev_B": np.zeros((B, H, 1, N), np.float32), "prev_x": np.zeros((B, H, 1, Pd), np.float32)}


def prior_h(B, H, N, Pd, dtype, seed, T0=96):
    st = P.prior_state(B, H, N, Pd, 1, dtype, seed, T0)
    return st["h"]


def ssd_prefill_gpu(inp, dtype, h0=None, out_dtype=torch.float32):
    d = P.to_device(inp, dtype)
    x = d["x"][:, :, :, 0].contiguous()
    Bm, Cm = d["B"][:, :, :, 0].contiguous(), d["C"][:, :, :, 0].contiguous()
    Bsz, T, H, Pd = x.shape
    N = Bm.shape[-1]
    hT = torch.zeros(Bsz, H, N, Pd, dtype=torch.float32, device="cuda")
    ws = m3.workspace_for(m3.M3Dims(Bsz, T, H, Pd, N, 1, 0, m3.M3_BF16 if dtype == "bf16" else m3.M3_F32,
                                    m3.M3_F32), "cuda")
    h0d = torch.from_numpy(h0).cuda() if h0 is not None else None
    y = m3.m3_ssd_prefill(x, Bm, Cm, d["dt"], d["A"], h0d, hT=hT, workspace=ws, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert m3.m3_ssm_device_status(ws) == m3.M3_OK
    return y, hT


def compare(y, hT, inp, h0, dtype, slices):
    N, Pd = inp["B"].shape[-1], inp["x"].shape[-1]
    B, H = inp["dt"].shape[0], inp["dt"].shape[2]
    st0 = ssd_state(h0, N, Pd) if h0 is not None else None
    yr, sr = P.run_oracle(inp, slices, st0)
    e = P.rel_err(P.pick(y.float().cpu().numpy(), slices, True), yr)
    assert e <= P.TOL[dtype], e
    eh = P.rel_err(P.pick(hT.cpu().numpy(), slices, False), sr["h"])
    assert eh <= P.TOL[dtype], eh


@pytest.mark.parametrize("N", [128, 64])
@pytest.mark.parametrize("fresh", [False, True])
def test_ssd_tensor_core_prefill(N, fresh):
    """tcgen05 path without the rotation: three full chunks plus a ragged tail."""
    B, H, Pd = 2, 3, 64
    T = 3 * 128 + 64 + 3
    inp = ssd_inputs(B, T, H, Pd, N, 5000 + N, "bf16")
    h0 = None if fresh else prior_h(B, H, N, Pd, "bf16", 23)
    y, hT = ssd_prefill_gpu(inp, "bf16", h0)
    compare(y, hT, inp, h0, "bf16", P.all_slices(B, H))


@pytest.mark.parametrize("fresh", [False, True])
def test_ssd_segmented_long_sequence_prefill(fresh):
    """Few (batch row, head) pairs and a long sequence: the segmented two-pass path."""
    B, H, Pd, N, T = 1, 4, 64, 128, 1500
    inp = ssd_inputs(B, T, H, Pd, N, 5100, "bf16")
    assert m3.m3_ssm_prefill_workspace(m3.M3Dims(B, T, H, Pd, N, 1, 0, m3.M3_BF16, m3.M3_F32)) > 256
    h0 = None if fresh else prior_h(B, H, N, Pd, "bf16", 29)
    y, hT = ssd_prefill_gpu(inp, "bf16", h0)
    compare(y, hT, inp, h0, "bf16", P.all_slices(B, H))


@pytest.mark.parametrize("N,Pd,T", [(16, 16, 40), (128, 64, 150), (6, 8, 1)])
def test_ssd_f32_recurrent_prefill(N, Pd, T):
    B, H = 2, 3
    inp = ssd_inputs(B, T, H, Pd, N, 5200 + N + T, "f32")
    h0 = P.random_state(B, H, N, Pd, 1, "f32", 31)["h"]
    y, hT = ssd_prefill_gpu(inp, "f32", h0)
    compare(y, hT, inp, h0, "f32", P.all_slices(B, H))


def test_ssd_bf16_output_and_in_place_continuation():
    """y in bf16; prefill(0:T1) then prefill(T1:T) with hT = h0 in place equals prefill(0:T)."""
    B, H, Pd, N, T, T1 = 2, 2, 64, 128, 400, 170
    inp = ssd_inputs(B, T, H, Pd, N, 5300, "bf16")
    first = {k: (v[:, :T1] if k != "A" else v) for k, v in inp.items()}
    second = {k: (v[:, T1:] if k != "A" else v) for k, v in inp.items()}
    _, h1 = ssd_prefill_gpu(first, "bf16")
    d = P.to_device(second, "bf16")
    x = d["x"][:, :, :, 0].contiguous()
    Bm, Cm = d["B"][:, :, :, 0].contiguous(), d["C"][:, :, :, 0].contiguous()
    y2 = m3.m3_ssd_prefill(x, Bm, Cm, d["dt"], d["A"], h1, hT=h1, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    sl = P.all_slices(B, H)
    yr, sr = P.run_oracle(inp, sl)
    # y rounded to bf16: the bound is the fp32-output tolerance plus one bf16 rounding (2^-8 |y|)
    got, ref = P.pick(y2.float().cpu().numpy(), sl, True), yr[:, T1:]
    rms = np.sqrt(np.mean(ref * ref))
    assert np.all(np.abs(got - ref) <= P.TOL["bf16"] * rms + 2.0 ** -8 * np.abs(ref))
    assert P.rel_err(P.pick(h1.cpu().numpy(), sl, False), sr["h"]) <= P.TOL["bf16"]


@pytest.mark.parametrize("N,dtype", [(128, "bf16"), (64, "bf16"), (32, "f32"), (128, "f32")])
def test_ssd_decode_steps_match_oracle(N, dtype):
    """Five decode steps from an entry state; every output and the final state."""
    B, H, Pd, steps = 3, 4, 64, 5
    inp = ssd_inputs(B, steps, H, Pd, N, 5400 + N, dtype)
    h0 = P.random_state(B, H, N, Pd, 1, "f32", 37)["h"] * 0.1
    d = P.to_device(inp, dtype)
    h = torch.from_numpy(h0).cuda()
    ys = []
    for t in range(steps):
        ys.append(m3.m3_ssd_decode_step(h, d["x"][:, t, :, 0].contiguous(), d["B"][:, t, :, 0].contiguous(),
                                        d["C"][:, t, :, 0].contiguous(), d["dt"][:, t].contiguous(),
                                        d["A"]).cpu().numpy())
    torch.cuda.synchronize()
    sl = P.all_slices(B, H)
    yr, sr = P.run_oracle(inp, sl, ssd_state(h0, N, Pd))
    y = np.stack(ys, axis=1)  # [B, steps, H, 1, P]
    e = P.rel_err(P.pick(y, sl, True), yr)
    assert e <= P.TOL[dtype], e
    assert P.rel_err(P.pick(h.cpu().numpy(), sl, False), sr["h"]) <= P.TOL[dtype]


def test_ssd_prefill_close_to_full_method_with_unit_lambda_zero_theta():
    """The special case and the full method fed lambda = 1, theta = 0 compute the same map."""
    B, H, Pd, N, T = 2, 3, 64, 128, 300
    inp = ssd_inputs(B, T, H, Pd, N, 5500, "bf16")
    y_ssd, h_ssd = ssd_prefill_gpu(inp, "bf16")
    d = P.to_device(inp, "bf16")
    st = m3.State.zeros(B, H, N, Pd, 1)
    y_full = m3.m3_ssm_prefill(d["x"], d["B"], d["C"], d["dt"], d["A"], d["lambda"], d["theta"],
                               hT=st)
    torch.cuda.synchronize()
    ref = y_full.float().cpu().numpy()
    assert P.rel_err(y_ssd.float().cpu().numpy(), ref) <= 2e-2
    assert P.rel_err(h_ssd.cpu().numpy(), st.h.cpu().numpy()) <= 2e-2


def test_ssd_full_size_sampled():
    """The benchmark's Mamba-2 comparison workloads at full size, in the benchmark's launch
    configuration: prefill B8 T4096 H32 N128 and one decode step at B256 H32 N128 from the
    prefill-sized state; sampled (b, h) sequences against the oracle."""
    w = synth.WORKLOADS["siso-prefill-bf16-b8-t4096-h32-p64-n128"]
    inp = ssd_inputs(w.B, w.T, w.H, w.P, w.N, w.seed, "bf16")
    y, hT = ssd_prefill_gpu(inp, "bf16")
    compare(y, hT, inp, None, "bf16", P.sample_slices(w.B, w.H, 6, 41))
    wd = synth.WORKLOADS["siso-decode-bf16-b256-h32-p64-n128"]
    dinp = ssd_inputs(wd.B, 1, wd.H, wd.P, wd.N, wd.seed, "bf16")
    h0 = P.random_state(wd.B, wd.H, wd.N, wd.P, 1, "f32", 43)["h"] * 0.05
    d = P.to_device(dinp, "bf16")
    h = torch.from_numpy(h0).cuda()
    yt = m3.m3_ssd_decode_step(h, d["x"][:, 0, :, 0].contiguous(), d["B"][:, 0, :, 0].contiguous(),
                               d["C"][:, 0, :, 0].contiguous(), d["dt"][:, 0].contiguous(), d["A"])
    torch.cuda.synchronize()
    sl = P.sample_slices(wd.B, wd.H, 16, 47)
    yr, sr = P.run_oracle(dinp, sl, ssd_state(h0, wd.N, wd.P))
    e = P.rel_err(P.pick(yt.cpu().numpy()[:, None], sl, True), yr)
    assert e <= P.TOL["bf16"], e
    assert P.rel_err(P.pick(h.cpu().numpy(), sl, False), sr["h"]) <= P.TOL["bf16"]
