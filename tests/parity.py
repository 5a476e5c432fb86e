"""Helpers shared by the GPU parity tests: move seeded inputs to the device, run the
oracle on the same (b, h) sequences, and measure the error the way the tolerance is
stated (max abs error over the compared elements divided by their RMS)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import state_space_sequence_trapezoidal_b300 as m3
from state_space_sequence_trapezoidal_b300 import synth

# Tolerances: max|gpu - oracle| / rms(oracle) for fp32 inputs and for bf16 inputs with
# fp32 accumulation (the target accuracy of the method's implementation).
TOL = {"f32": 1e-4, "bf16": 2e-2}
# Angle carried in the state, compared modulo 2 pi.
PHI_TOL = {"f32": 1e-4, "bf16": 2e-3}


def tdtype(dtype: str):
    return torch.bfloat16 if dtype == "bf16" else torch.float32


def to_device(inp: dict, dtype: str, device="cuda") -> dict:
    out = {}
    for k, v in inp.items():
        out[k] = torch.from_numpy(np.ascontiguousarray(v)).to(
            device=device, dtype=torch.float32 if k == "A" else tdtype(dtype))
    return out


def random_state(B, H, N, P, R, dtype: str, seed: int) -> dict:
    """A non-trivial entry state (numpy, values exact in the state dtypes)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    st = {
        "h": rng.standard_normal((B, H, N, P)).astype(np.float32),
        "phi": rng.uniform(-3, 3, (B, H, N // 2)).astype(np.float32),
        "prev_B": (rng.standard_normal((B, H, R, N)) / np.sqrt(N * R)).astype(np.float32),
        "prev_x": rng.standard_normal((B, H, R, P)).astype(np.float32),
    }
    if dtype == "bf16":
        st["prev_B"] = synth.round_bf16(st["prev_B"])
        st["prev_x"] = synth.round_bf16(st["prev_x"])
    return st


def prior_state(B, H, N, P, R, dtype: str, seed: int, T0: int = 96) -> dict:
    """An entry state of the kind a previous call hands over: the oracle's exit state after
    T0 seeded tokens from rest (h, the unreduced angle, the raw last token).  Its magnitude
    is that of the states the recurrence itself produces on these input distributions."""
    inp = synth.make_inputs(B, T0, H, P, N, R, seed, dtype)
    g = oracle.gather(inp, all_slices(B, H))
    _, st, _ = oracle.scan(g["x"], g["Bm"], g["Cm"], g["dt"], g["A"], g["lam"], g["theta"])
    out = {k: np.zeros((B, H) + v.shape[1:], np.float32) for k, v in st.items()}
    for i, (b, h) in enumerate(all_slices(B, H)):
        for k in st:
            out[k][b, h] = st[k][i]
    return out


def state_to_device(st: dict, dtype: str, device="cuda") -> m3.State:
    return m3.State(torch.from_numpy(st["h"]).to(device),
                    torch.from_numpy(st["phi"]).to(device),
                    torch.from_numpy(st["prev_B"]).to(device=device, dtype=tdtype(dtype)),
                    torch.from_numpy(st["prev_x"]).to(device=device, dtype=tdtype(dtype)))


def state_to_host(s: m3.State) -> dict:
    return {"h": s.h.float().cpu().numpy(), "phi": s.phi.float().cpu().numpy(),
            "prev_B": s.prev_B.float().cpu().numpy(), "prev_x": s.prev_x.float().cpu().numpy()}


def all_slices(B, H):
    return [(b, h) for b in range(B) for h in range(H)]


def sample_slices(B, H, n, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    idx = rng.choice(B * H, size=min(n, B * H), replace=False)
    return [(int(i) // H, int(i) % H) for i in sorted(idx)]


def run_oracle(inp: dict, slices, state: dict | None = None, nthreads: int = 0):
    layout = dict(inp)
    if state is not None:
        layout["state"] = state
    g = oracle.gather(layout, slices)
    y, st, _ = oracle.scan(g["x"], g["Bm"], g["Cm"], g["dt"], g["A"], g["lam"], g["theta"],
                           state=g.get("state"), nthreads=nthreads)
    return y, st


def pick(a: np.ndarray, slices, seq_axis: bool) -> np.ndarray:
    """Stack (b, h) sequences: [B,T,H,...] -> [S,T,...] (seq_axis) or [B,H,...] -> [S,...]."""
    if seq_axis:
        return np.stack([a[b, :, h] for b, h in slices])
    return np.stack([a[b, h] for b, h in slices])


def rel_err(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref * ref))
    return float(np.max(np.abs(got - ref)) / max(rms, 1e-30))


def phi_err(got, ref) -> float:
    d = np.asarray(got, np.float64) - np.asarray(ref, np.float64)
    d = (d + np.pi) % (2 * np.pi) - np.pi
    return float(np.max(np.abs(d))) if d.size else 0.0


def check_state(got: dict, ref: dict, dtype: str, what=""):
    e = rel_err(got["h"], ref["h"])
    assert e <= TOL[dtype], f"{what} h_T: rel err {e:.3g} > {TOL[dtype]}"
    pe = phi_err(got["phi"], ref["phi"])
    assert pe <= PHI_TOL[dtype], f"{what} phi_T: err {pe:.3g}"
    np.testing.assert_array_equal(got["prev_B"], ref["prev_B"].astype(np.float32))
    np.testing.assert_array_equal(got["prev_x"], ref["prev_x"].astype(np.float32))
