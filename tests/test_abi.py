"""The C-ABI library loads, exports every function include/m3_ssm.h declares, and
rejects bad arguments on the host before anything reaches a GPU.

None of these calls launches a kernel: each one fails validation first."""
import ctypes
import glob
import os
import re

import pytest

import state_space_sequence_trapezoidal_b300 as m3
from state_space_sequence_trapezoidal_b300 import M3Dims, M3State

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

OK, ARG, SHAPE, DTYPE, ALIGN, CUDA, TIMEOUT, UNSUP, WS, RANGE = range(10)


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(m3_\w+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported():
    lib = m3.load()
    names = declared_functions()
    assert {"m3_ssm_prefill", "m3_ssm_decode_step", "m3_ssm_prefill_workspace",
            "m3_ssm_device_status", "m3_status_str"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported by libm3ssm.so"


def test_status_strings():
    lib = m3.load()
    for s in range(10):
        assert lib.m3_status_str(s)
    assert lib.m3_status_str(99) == b"unknown status"


def _dims(**kw):
    d = dict(B=2, T=8, H=3, P=64, N=128, R=1, chunk=0, in_dtype=1, out_dtype=0)
    d.update(kw)
    return M3Dims(**d)


def _prefill(d, ptrs=None, ws=256, h0=None, hT=None):
    lib = m3.load()
    p = dict(x=16, B=16, C=16, dt=16, A=16, lam=16, theta=16, y=16, ws=16)
    p.update(ptrs or {})
    return lib.m3_ssm_prefill(ctypes.byref(d) if d is not None else None, p["x"], p["B"], p["C"],
                              p["dt"], p["A"], p["lam"], p["theta"],
                              ctypes.byref(h0) if h0 else None, p["y"],
                              ctypes.byref(hT) if hT else None, p["ws"], ws, None)


@pytest.mark.parametrize("kw,code", [
    (dict(N=127), SHAPE), (dict(N=0), SHAPE), (dict(N=258), SHAPE), (dict(P=6), SHAPE),
    (dict(P=0), SHAPE), (dict(R=3), SHAPE), (dict(B=-1), SHAPE), (dict(T=-1), SHAPE),
    (dict(chunk=-1), SHAPE), (dict(in_dtype=7), DTYPE), (dict(out_dtype=5), DTYPE),
])
def test_prefill_rejects_bad_dims(kw, code):
    assert _prefill(_dims(**kw)) == code


def test_prefill_rejects_null_and_misaligned_pointers():
    assert _prefill(None) == ARG
    assert _prefill(_dims(), dict(x=None)) == ARG
    assert _prefill(_dims(), dict(A=None)) == ARG
    assert _prefill(_dims(), dict(ws=None)) == WS
    assert _prefill(_dims(), ws=8) == WS
    assert _prefill(_dims(), dict(theta=24)) == ALIGN
    assert _prefill(_dims(), dict(y=4)) == ALIGN
    partial = M3State(16, None, 16, 16)
    assert _prefill(_dims(), h0=partial) == ARG
    assert _prefill(_dims(), hT=M3State(16, 16, 16, 8)) == ALIGN


def test_workspace_size():
    assert m3.m3_ssm_prefill_workspace(_dims()) >= 256
    # a long sequence over few (batch row, head) pairs is split into segments, whose
    # per-segment states live in the workspace
    long = _dims(B=1, T=16384, H=32)
    assert m3.m3_ssm_prefill_workspace(long) > 1 << 20
    assert m3.m3_ssm_prefill_workspace(_dims(B=1, T=16384, H=32, in_dtype=0)) == 256


def test_bcnorm_entry_points_reject_bad_arguments():
    """The fused BCNorm calls: norm required, eps > 0 and finite, parameters 16-byte aligned."""
    lib = m3.load()
    from state_space_sequence_trapezoidal_b300 import M3BcNorm

    def pre(d, norm, x=16):
        return lib.m3_ssm_prefill_bcnorm(ctypes.byref(d), x, 16, 16, 16, 16, 16, 16,
                                         ctypes.byref(norm) if norm else None, None, 16, None,
                                         16, 256, None)

    def dec(d, norm, x=16):
        st = M3State(16, 16, 16, 16)
        return lib.m3_ssm_decode_step_bcnorm(ctypes.byref(d), ctypes.byref(st), x, 16, 16, 16, 16,
                                             16, 16, ctypes.byref(norm) if norm else None, 16, None)

    good = M3BcNorm(16, 32, None, 48, 1e-5)
    for call in (pre, dec):
        assert call(_dims(), None) == ARG
        assert call(_dims(), M3BcNorm(16, 16, 16, 16, 0.0)) == ARG
        assert call(_dims(), M3BcNorm(16, 16, 16, 16, -1.0)) == ARG
        assert call(_dims(), M3BcNorm(16, 16, 16, 16, float("inf"))) == ARG
        assert call(_dims(), M3BcNorm(16, 24, 16, 16, 1e-5)) == ALIGN
        assert call(_dims(N=7), good) == SHAPE
        assert call(_dims(), good, x=None) == ARG
        assert call(_dims(), good, x=8) == ALIGN


def test_decode_rejects_bad_arguments():
    lib = m3.load()
    st = M3State(16, 16, 16, 16)

    def call(d, state=st, x=16):
        return lib.m3_ssm_decode_step(ctypes.byref(d), ctypes.byref(state) if state else None,
                                      x, 16, 16, 16, 16, 16, 16, 16, None)

    assert call(_dims(N=5)) == SHAPE
    assert call(_dims(R=5)) == SHAPE
    assert call(_dims(), state=None) == ARG
    assert call(_dims(), x=None) == ARG
    assert call(_dims(), x=40) == ALIGN
    assert call(_dims(), state=M3State(16, 16, None, 16)) == ARG


def test_ssd_entry_points_reject_bad_arguments():
    """The Mamba-2 special case: SISO only, lambda/theta absent, state h alone."""
    lib = m3.load()

    def pre(d, x=16, h0=None, hT=None, ws=16, wsb=256, y=16):
        return lib.m3_ssd_prefill(ctypes.byref(d), x, 16, 16, 16, 16, h0, y, hT, ws, wsb, None)

    def dec(d, h=16, x=16, y=16):
        return lib.m3_ssd_decode_step(ctypes.byref(d), h, x, 16, 16, 16, 16, y, None)

    assert pre(_dims(R=2)) == SHAPE
    assert pre(_dims(N=7)) == SHAPE
    assert pre(_dims(), x=None) == ARG
    assert pre(_dims(), ws=None) == WS
    assert pre(_dims(), wsb=8) == WS
    assert pre(_dims(), y=8) == ALIGN
    assert pre(_dims(), h0=24) == ALIGN
    assert pre(_dims(), hT=40) == ALIGN
    assert dec(_dims(R=4)) == SHAPE
    assert dec(_dims(), h=None) == ARG
    assert dec(_dims(), x=None) == ARG
    assert dec(_dims(), h=8) == ALIGN
    assert dec(_dims(), y=4) == ALIGN


def test_backward_rejects_bad_arguments():
    lib = m3.load()

    def call(d, x=16, dy=16, dx=16, dA=16, ws=16, wsb=1 << 30, dhT=None, dh0=None):
        return lib.m3_ssm_prefill_backward(ctypes.byref(d), x, 16, 16, 16, 16, 16, 16, None, dy, dhT,
                                           dx, 16, 16, 16, dA, 16, 16, dh0, ws, wsb, None)

    assert call(_dims(N=7)) == SHAPE
    assert call(_dims(N=256, P=64)) == SHAPE          # N P > 8192: not supported
    assert call(_dims(), ws=None) == WS
    assert call(_dims(), wsb=8) == WS
    assert call(_dims(), x=None) == ARG
    assert call(_dims(), dy=None) == ARG
    assert call(_dims(), dA=None) == ARG
    assert call(_dims(), dx=8) == ALIGN
    assert call(_dims(), dhT=24) == ALIGN
    assert call(_dims(), dh0=40) == ALIGN


def test_backward_workspace_holds_the_chunk_states():
    lib = m3.load()
    d = _dims(B=8, T=4096, H=32, P=64, N=128)
    n = lib.m3_ssm_prefill_backward_workspace(ctypes.byref(d))
    # per (batch row, head) and chunk of 32 tokens: the folded entry state and the exit
    # cotangent, N x P floats each
    assert n >= 2 * 8 * 32 * (4096 // 32) * 128 * 64 * 4
    assert lib.m3_ssm_prefill_backward_workspace(ctypes.byref(_dims(N=256, P=64))) == 256


def test_backward_refuses_state_wider_than_1024():
    lib = m3.load()
    d = _dims(N=2048, P=4)  # N P = 8192 fits, but N / 2 pairs exceed the kernels' 512 threads
    assert lib.m3_ssm_prefill_backward_workspace(ctypes.byref(d)) == 256
    dd = _dims(N=2048, P=4)
    assert lib.m3_ssm_prefill_backward(ctypes.byref(dd), 16, 16, 16, 16, 16, 16, 16, None, 16, None,
                                       16, 16, 16, 16, 16, 16, 16, None, 16, 1 << 30, None) == SHAPE


@pytest.mark.parametrize("R,c", [(1, 32), (2, 32), (4, 16), (8, 8)])
def test_backward_chunk_length_per_rank(R, c):
    """Chunks of 32 tokens while c R <= 64 (token, rank) rows, halved beyond: the workspace holds
    two N x P fp32 states per chunk, plus per-chunk scalars and angle sums and one state per
    sequence."""
    lib = m3.load()
    Bsz, T, H, N, P = 2, 1000, 3, 64, 64
    d = _dims(B=Bsz, T=T, H=H, P=P, N=N, R=R)
    n = lib.m3_ssm_prefill_backward_workspace(ctypes.byref(d))
    bh, nch, K = Bsz * H, -(-T // c), N // 2
    states = 2 * bh * nch * N * P * 4
    rest = (bh * nch * (3 + 2 * K) + bh * N * P + bh) * 4 + 10 * 256
    assert states <= n <= states + rest, (n, states, rest)
