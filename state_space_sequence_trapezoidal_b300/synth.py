"""Seeded synthetic inputs for the Mamba-3 SSM core.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic, so both the CUDA path's tests/benchmark and the oracle
can take their inputs from it.

Distributions follow the 1.5B-scale layer workloads the paper benchmarks
(section 4.4: d_model 2048, state sizes 64/128, batch 128 decode; 16384-token
sequences): x ~ N(0, 1); B, C ~ N(0, 1/(N R)); dt = softplus(N(-2, 0.5));
A = -exp(U(0, ln 16)) per head; lambda = sigmoid(N(0, 1));
theta ~ N(0, 1) per rotation pair.  Values are rounded to nearest-even in
the requested input dtype on the host, so the device and the oracle see
identical numbers.  A stays float32.

Layouts (innermost index last): x [B,T,H,R,P]; B, C [B,T,H,R,N];
dt, lambda [B,T,H]; theta [B,T,H,N/2]; A [H].
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); return float32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    P: int
    N: int
    R: int
    dtype: str  # "f32" or "bf16"
    seed: int
    decode_steps: int = 0  # decode steps that follow the prefill (0: prefill only)
    prefill_T_for_decode: int = 0


# The five workloads of the benchmark plan, named by what they are.
WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny-siso-f32-b1-h2-t256-p16-n16", 1, 256, 2, 16, 16, 1, "f32", 20260000),
        Workload("siso-prefill-bf16-b8-t4096-h32-p64-n128", 8, 4096, 32, 64, 128, 1, "bf16", 20260001),
        Workload("mimo-r4-prefill-bf16-b8-t4096-h32-p64-n64", 8, 4096, 32, 64, 64, 4, "bf16", 20260002),
        Workload("siso-decode-bf16-b256-h32-p64-n128", 256, 1, 32, 64, 128, 1, "bf16", 20260003,
                 decode_steps=1000, prefill_T_for_decode=512),
        Workload("mimo-r4-decode-bf16-b256-h32-p64-n64", 256, 1, 32, 64, 64, 4, "bf16", 20260003,
                 decode_steps=1000, prefill_T_for_decode=512),
        Workload("long-siso-prefill-bf16-b1-t16384-h32-p64-n128", 1, 16384, 32, 64, 128, 1, "bf16",
                 20260004, decode_steps=256),
    ]
}


def make_inputs(B: int, T: int, H: int, P: int, N: int, R: int, seed: int, dtype: str = "bf16",
                A_seed: int | None = None) -> dict:
    """Draw one batch of inputs.  Returns float32 numpy arrays (bf16-exact if dtype == "bf16").

    ``A_seed`` (default: ``seed``) seeds the per-head A separately, so that a
    decode loop can draw fresh per-token inputs every step with the same A.
    """
    assert N % 2 == 0
    rng = np.random.Generator(np.random.PCG64(seed))
    f32 = np.float32
    x = rng.standard_normal((B, T, H, R, P), dtype=f32)
    sd = f32(1.0 / np.sqrt(N * R))
    Bm = rng.standard_normal((B, T, H, R, N), dtype=f32) * sd
    Cm = rng.standard_normal((B, T, H, R, N), dtype=f32) * sd
    z = rng.normal(-2.0, 0.5, size=(B, T, H)).astype(f32)
    dt = np.logaddexp(f32(0), z).astype(f32)  # softplus
    lam = (1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, H), dtype=f32)))).astype(f32)
    theta = rng.standard_normal((B, T, H, N // 2), dtype=f32)
    arng = np.random.Generator(np.random.PCG64(seed if A_seed is None else A_seed))
    A = (-np.exp(arng.uniform(0.0, np.log(16.0), size=H))).astype(f32)
    out = {"x": x, "B": Bm, "C": Cm, "dt": dt, "lambda": lam, "theta": theta, "A": A}
    if dtype == "bf16":
        for k in ("x", "B", "C", "dt", "lambda", "theta"):
            out[k] = round_bf16(out[k])
    elif dtype != "f32":
        raise ValueError(f"unknown dtype {dtype!r}")
    return out


def decode_step_seed(base_seed: int, step: int) -> int:
    """Seed of the per-token inputs of decode step ``step`` (0-based)."""
    return base_seed + 100 + step


def make_raw_bc(inp: dict, seed: int, dtype: str = "bf16") -> dict:
    """Raw B, C projection outputs for the BCNorm entry points: the drawn B and C with every
    (token, head, rank) row scaled by its own random factor exp(N(0, 1)) (so the normalisation
    has work to do), rounded to the input dtype.  Returns a copy of ``inp`` with B, C replaced."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = dict(inp)
    for k in ("B", "C"):
        sc = np.exp(rng.standard_normal(inp[k].shape[:-1] + (1,), dtype=np.float32))
        v = (inp[k] * sc).astype(np.float32)
        out[k] = round_bf16(v) if dtype == "bf16" else v
    return out


def make_bcnorm_params(N: int, H: int, R: int, seed: int, dtype: str = "bf16") -> dict:
    """BCNorm weights [N] ~ U(0.5, 1.5) / sqrt(N R) and biases [H, N] ~ N(0, 0.09 / (N R)) for B
    and for C, so that the normalised B, C have about the scale of the drawn ones; rounded to
    the input dtype.  eps = 1e-5."""
    rng = np.random.Generator(np.random.PCG64(seed))
    s = np.float32(1.0 / np.sqrt(N * R))
    p = {"B_weight": rng.uniform(0.5, 1.5, N).astype(np.float32) * s,
         "B_bias": (0.3 * rng.standard_normal((H, N))).astype(np.float32) * s,
         "C_weight": rng.uniform(0.5, 1.5, N).astype(np.float32) * s,
         "C_bias": (0.3 * rng.standard_normal((H, N))).astype(np.float32) * s}
    if dtype == "bf16":
        p = {k: round_bf16(v) for k, v in p.items()}
    p["eps"] = 1e-5
    return p
