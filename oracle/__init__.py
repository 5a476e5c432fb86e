"""Oracle for the Mamba-3 SSM layer core -- test infrastructure, not product.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg may import this package.  The CUDA path never does, and this
package never touches the CUDA path: the two share no code.

``m3_oracle.c`` holds the sequential fp64 recurrence (its header cites the
paper passages it follows).  This module compiles it with gcc on first use,
and marshals numpy arrays in and out.  Every input is upcast exactly to
float64 before the call (bf16 and fp32 values are exact in fp64).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "m3_oracle.c")
_LIB = os.path.join(_HERE, "libm3oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/libm3oracle.so`` (gcc, -O2, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            i = ctypes.c_int
            lib.m3o_scan_batch.argtypes = [i] * 5 + [dp] * 12 + [i]
            lib.m3o_scan_batch.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def zero_state(S: int, N: int, P: int, R: int) -> dict:
    return {
        "h": np.zeros((S, N, P)),
        "phi": np.zeros((S, N // 2)),
        "prev_B": np.zeros((S, R, N)),
        "prev_x": np.zeros((S, R, P)),
    }


def scan(x, Bm, Cm, dt, A, lam, theta, state: dict | None = None, nthreads: int = 0):
    """Run the recurrence on S independent sequences.

    Shapes (S sequences, T tokens): x [S,T,R,P]; Bm, Cm [S,T,R,N]; dt, lam [S,T];
    A [S]; theta [S,T,N/2]; state {h [S,N,P], phi [S,N/2], prev_B [S,R,N],
    prev_x [S,R,P]} or None for a fresh start.
    Returns (y [S,T,R,P] float64, final state dict, threads used).
    """
    x = _f64(x)
    S, T, R, P = x.shape
    Bm, Cm = _f64(Bm), _f64(Cm)
    N = Bm.shape[-1]
    assert Bm.shape == (S, T, R, N) and Cm.shape == (S, T, R, N)
    assert N % 2 == 0
    dt, lam = _f64(dt).reshape(S, T), _f64(lam).reshape(S, T)
    theta = _f64(theta).reshape(S, T, N // 2)
    A = _f64(A).reshape(S)
    st = zero_state(S, N, P, R) if state is None else {k: _f64(v).copy() for k, v in state.items()}
    st["h"] = st["h"].reshape(S, N, P).copy()
    st["phi"] = st["phi"].reshape(S, N // 2).copy()
    st["prev_B"] = st["prev_B"].reshape(S, R, N).copy()
    st["prev_x"] = st["prev_x"].reshape(S, R, P).copy()
    y = np.zeros((S, T, R, P))
    used = _load().m3o_scan_batch(
        S, T, N, P, R, _ptr(x), _ptr(Bm), _ptr(Cm), _ptr(dt), _ptr(A), _ptr(lam), _ptr(theta),
        _ptr(st["h"]), _ptr(st["phi"]), _ptr(st["prev_B"]), _ptr(st["prev_x"]), _ptr(y), nthreads,
    )
    return y, st, used


def gather(layout: dict, slices) -> dict:
    """Pick (b, h) sequences out of arrays in the library's [B,T,H,...] layout.

    ``layout`` holds x [B,T,H,R,P], B/C [B,T,H,R,N], dt/lambda [B,T,H],
    A [H], theta [B,T,H,N/2] (numpy or anything np.asarray accepts) and,
    optionally, a state {h [B,H,N,P], phi [B,H,N/2], prev_B [B,H,R,N],
    prev_x [B,H,R,P]}.  Returns the per-sequence stacks ``scan`` takes.
    """
    bs = [b for b, _ in slices]
    hs = [h for _, h in slices]

    def seq(a):
        a = np.asarray(a)
        return np.stack([a[b, :, h] for b, h in zip(bs, hs)])

    out = {
        "x": seq(layout["x"]),
        "Bm": seq(layout["B"]),
        "Cm": seq(layout["C"]),
        "dt": seq(layout["dt"]),
        "lam": seq(layout["lambda"]),
        "theta": seq(layout["theta"]),
        "A": np.asarray(layout["A"])[hs],
    }
    if layout.get("state") is not None:
        s = layout["state"]
        out["state"] = {k: np.stack([np.asarray(s[k])[b, h] for b, h in zip(bs, hs)])
                        for k in ("h", "phi", "prev_B", "prev_x")}
    return out
