"""ctypes binding of ``libm3ssm.so`` (declared in ``include/m3_ssm.h``).

Argument marshalling only: torch supplies device memory and streams, and every
step of the computation runs in the library's CUDA kernels.  There is no
fallback: if the library cannot be loaded, or a call returns an error status,
the functions here raise.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import torch

from . import build as _build

M3_OK = 0
M3_ERR_TIMEOUT = 6
M3_ERR_UNSUPPORTED = 7
M3_ERR_WORKSPACE = 8
M3_ERR_RANGE = 9
M3_F32, M3_BF16 = 0, 1
_DT = {torch.float32: M3_F32, torch.bfloat16: M3_BF16}


class M3Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("B", "T", "H", "P", "N", "R", "chunk", "in_dtype", "out_dtype")]


class M3State(ctypes.Structure):
    _fields_ = [("h", ctypes.c_void_p), ("phi", ctypes.c_void_p), ("prev_B", ctypes.c_void_p),
                ("prev_x", ctypes.c_void_p)]


class M3BcNorm(ctypes.Structure):
    _fields_ = [("B_weight", ctypes.c_void_p), ("B_bias", ctypes.c_void_p),
                ("C_weight", ctypes.c_void_p), ("C_bias", ctypes.c_void_p),
                ("eps", ctypes.c_float)]


class M3Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: m3 status {status} ({status_str(status)})")


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libm3ssm.so (building it first if the sources are newer)."""
    global _lib
    with _lock:
        if _lib is None:
            if _build.needs_build():
                _build.build()
            lib = ctypes.CDLL(_build.LIB)
            vp, sz = ctypes.c_void_p, ctypes.c_size_t
            dp, sp = ctypes.POINTER(M3Dims), ctypes.POINTER(M3State)
            lib.m3_ssm_prefill_workspace.argtypes = [dp]
            lib.m3_ssm_prefill_workspace.restype = sz
            lib.m3_ssm_prefill.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, sp, vp, sp, vp, sz, vp]
            lib.m3_ssm_prefill.restype = ctypes.c_int
            lib.m3_ssm_prefill_noalloc.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, sp, vp, sp, vp]
            lib.m3_ssm_prefill_noalloc.restype = ctypes.c_int
            lib.m3_ssm_decode_step.argtypes = [dp, sp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
            lib.m3_ssm_decode_step.restype = ctypes.c_int
            np_ = ctypes.POINTER(M3BcNorm)
            lib.m3_ssm_prefill_bcnorm.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, np_, sp, vp, sp,
                                                  vp, sz, vp]
            lib.m3_ssm_prefill_bcnorm.restype = ctypes.c_int
            lib.m3_ssm_decode_step_bcnorm.argtypes = [dp, sp, vp, vp, vp, vp, vp, vp, vp, np_, vp,
                                                      vp]
            lib.m3_ssm_decode_step_bcnorm.restype = ctypes.c_int
            lib.m3_ssm_prefill_backward_workspace.argtypes = [dp]
            lib.m3_ssm_prefill_backward_workspace.restype = sz
            lib.m3_ssm_prefill_backward.argtypes = [dp] + [vp] * 7 + [sp] + [vp] * 10 + [vp, sz, vp]
            lib.m3_ssm_prefill_backward.restype = ctypes.c_int
            lib.m3_ssd_prefill.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
            lib.m3_ssd_prefill.restype = ctypes.c_int
            lib.m3_ssd_decode_step.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp]
            lib.m3_ssd_decode_step.restype = ctypes.c_int
            lib.m3_ssm_device_status.argtypes = [vp, vp]
            lib.m3_ssm_device_status.restype = ctypes.c_int
            lib.m3_status_str.argtypes = [ctypes.c_int]
            lib.m3_status_str.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def status_str(status: int) -> str:
    return load().m3_status_str(int(status)).decode()


@dataclass
class State:
    """Recurrent state of the SSM core for B x H sequences.

    h [B,H,N,P] float32; phi [B,H,N/2] float32 (cumulative angle of the last
    token, kept reduced to [-pi, pi]); prev_B [B,H,R,N] and prev_x [B,H,R,P]
    in the input dtype (the last token's raw B and x).
    """

    h: torch.Tensor
    phi: torch.Tensor
    prev_B: torch.Tensor
    prev_x: torch.Tensor

    @staticmethod
    def zeros(B, H, N, P, R=1, dtype=torch.bfloat16, device="cuda") -> "State":
        return State(torch.zeros(B, H, N, P, dtype=torch.float32, device=device),
                     torch.zeros(B, H, N // 2, dtype=torch.float32, device=device),
                     torch.zeros(B, H, R, N, dtype=dtype, device=device),
                     torch.zeros(B, H, R, P, dtype=dtype, device=device))

    def clone(self) -> "State":
        return State(self.h.clone(), self.phi.clone(), self.prev_B.clone(), self.prev_x.clone())

    def _c(self) -> M3State:
        for t in (self.h, self.phi, self.prev_B, self.prev_x):
            if not t.is_contiguous():
                raise ValueError("state tensors must be contiguous")
        return M3State(self.h.data_ptr(), self.phi.data_ptr(), self.prev_B.data_ptr(),
                       self.prev_x.data_ptr())


@dataclass
class BCNorm:
    """BCNorm and the B, C biases applied by the *_bcnorm entry points: per (token, head,
    rank) vector v of N raw projection outputs, v / sqrt(mean(v^2) + eps) * weight + bias[h].
    Weights [N] and biases [H, N] in the input dtype, on the device; None = ones / zeros."""

    B_weight: torch.Tensor | None = None
    B_bias: torch.Tensor | None = None
    C_weight: torch.Tensor | None = None
    C_bias: torch.Tensor | None = None
    eps: float = 1e-6

    def _c(self, dtype, device, N: int, H: int) -> M3BcNorm:
        ptrs = []
        for name, shape in (("B_weight", (N,)), ("B_bias", (H, N)), ("C_weight", (N,)),
                            ("C_bias", (H, N))):
            t = getattr(self, name)
            if t is None:
                ptrs.append(None)
                continue
            if (t.dtype != dtype or t.device != device or not t.is_contiguous()
                    or tuple(t.shape) != shape):
                raise ValueError(f"{name}: {dtype} {list(shape)} contiguous on {device} expected")
            ptrs.append(t.data_ptr())
        return M3BcNorm(*ptrs, float(self.eps))


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check_inputs(ts, dtype):
    dev = None
    for name, t in ts.items():
        if t.dtype != dtype:
            raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
        if not t.is_cuda:
            raise ValueError(f"{name}: must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name}: must be contiguous")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"{name}: on {t.device}, others on {dev}")
    return dev


def _dims(x, dt, theta, chunk, in_dt, out_dt, prefill=True) -> M3Dims:
    if prefill:
        Bsz, T, H = dt.shape
    else:
        (Bsz, H), T = dt.shape, 0
    N = theta.shape[-1] * 2
    P = x.shape[-1]
    R = x.shape[-2] if x.dim() == (5 if prefill else 4) else 1
    return M3Dims(Bsz, T, H, P, N, R, chunk, _DT[in_dt], _DT[out_dt])


def m3_ssm_prefill_workspace(dims: M3Dims) -> int:
    return int(load().m3_ssm_prefill_workspace(ctypes.byref(dims)))


def workspace_for(dims: M3Dims, device) -> torch.Tensor:
    """A zero-filled workspace tensor for m3_ssm_prefill with these dimensions (the size
    depends on the SM count of the current device)."""
    n = m3_ssm_prefill_workspace(dims)
    return torch.zeros((n + 15) // 16 * 16, dtype=torch.uint8, device=device)


def prefill_workspace(x, dt, theta, out_dtype=torch.float32) -> torch.Tensor:
    """A zero-filled workspace for m3_ssm_prefill on inputs shaped like these."""
    return workspace_for(_dims(x, dt, theta, 0, x.dtype, out_dtype), x.device)


def m3_ssm_prefill(x, B, C, dt, A, lam, theta, h0: State | None = None, *, y=None,
                   hT: State | None = None, workspace=None, chunk: int = 0,
                   out_dtype=torch.float32, stream=None):
    """Chunked prefill.  x [B,T,H,R,P] (or [B,T,H,P] for R = 1), B/C [B,T,H,R,N]
    (or [B,T,H,N]), dt/lam [B,T,H], A [H] float32, theta [B,T,H,N/2].
    Returns y [B,T,H,R,P] in ``out_dtype`` (or writes the given ``y``).
    ``hT`` (optional) receives the exit state; it may be ``h0`` itself."""
    in_dt = x.dtype
    dev = _check_inputs(dict(x=x, B=B, C=C, dt=dt, lam=lam, theta=theta), in_dt)
    _check_inputs(dict(A=A), torch.float32)
    d = _dims(x, dt, theta, chunk, in_dt, out_dtype)
    if y is None:
        y = torch.empty(d.B, d.T, d.H, d.R, d.P, dtype=out_dtype, device=dev)
    elif y.dtype != out_dtype or not y.is_contiguous() or y.numel() != d.B * d.T * d.H * d.R * d.P:
        raise ValueError("y: wrong dtype, layout or size")
    if workspace is None:
        workspace = workspace_for(d, dev)
    c0 = h0._c() if h0 is not None else None
    c1 = hT._c() if hT is not None else None
    st = load().m3_ssm_prefill(ctypes.byref(d), x.data_ptr(), B.data_ptr(), C.data_ptr(),
                               dt.data_ptr(), A.data_ptr(), lam.data_ptr(), theta.data_ptr(),
                               ctypes.byref(c0) if c0 is not None else None, y.data_ptr(),
                               ctypes.byref(c1) if c1 is not None else None,
                               workspace.data_ptr(), workspace.numel(), _stream_handle(stream))
    if st != M3_OK:
        raise M3Error(st, "m3_ssm_prefill")
    return y


def m3_ssm_prefill_bcnorm(x, B_raw, C_raw, dt, A, lam, theta, norm: BCNorm,
                          h0: State | None = None, *, y=None, hT: State | None = None,
                          workspace=None, chunk: int = 0, out_dtype=torch.float32, stream=None):
    """m3_ssm_prefill on raw B, C projection outputs, with BCNorm and the biases (``norm``)
    applied inside the kernels.  The state's prev_B holds the raw previous B."""
    in_dt = x.dtype
    dev = _check_inputs(dict(x=x, B=B_raw, C=C_raw, dt=dt, lam=lam, theta=theta), in_dt)
    _check_inputs(dict(A=A), torch.float32)
    d = _dims(x, dt, theta, chunk, in_dt, out_dtype)
    nc = norm._c(in_dt, dev, d.N, d.H)
    if y is None:
        y = torch.empty(d.B, d.T, d.H, d.R, d.P, dtype=out_dtype, device=dev)
    elif y.dtype != out_dtype or not y.is_contiguous() or y.numel() != d.B * d.T * d.H * d.R * d.P:
        raise ValueError("y: wrong dtype, layout or size")
    if workspace is None:
        workspace = workspace_for(d, dev)
    c0 = h0._c() if h0 is not None else None
    c1 = hT._c() if hT is not None else None
    st = load().m3_ssm_prefill_bcnorm(ctypes.byref(d), x.data_ptr(), B_raw.data_ptr(),
                                      C_raw.data_ptr(), dt.data_ptr(), A.data_ptr(),
                                      lam.data_ptr(), theta.data_ptr(), ctypes.byref(nc),
                                      ctypes.byref(c0) if c0 is not None else None, y.data_ptr(),
                                      ctypes.byref(c1) if c1 is not None else None,
                                      workspace.data_ptr(), workspace.numel(),
                                      _stream_handle(stream))
    if st != M3_OK:
        raise M3Error(st, "m3_ssm_prefill_bcnorm")
    return y


def m3_ssm_decode_step_bcnorm(state: State, x_t, B_raw_t, C_raw_t, dt_t, A, lam_t, theta_t,
                              norm: BCNorm, *, y_t=None, out_dtype=torch.float32, stream=None):
    """m3_ssm_decode_step on raw B_t, C_t, with BCNorm and the biases applied in the step's
    prologue.  The state's prev_B holds (and receives) the raw B."""
    in_dt = x_t.dtype
    dev = _check_inputs(dict(x_t=x_t, B_t=B_raw_t, C_t=C_raw_t, dt_t=dt_t, lam_t=lam_t,
                             theta_t=theta_t), in_dt)
    _check_inputs(dict(A=A), torch.float32)
    d = _dims(x_t, dt_t, theta_t, 0, in_dt, out_dtype, prefill=False)
    nc = norm._c(in_dt, dev, d.N, d.H)
    if y_t is None:
        y_t = torch.empty(d.B, d.H, d.R, d.P, dtype=out_dtype, device=dev)
    c = state._c()
    st = load().m3_ssm_decode_step_bcnorm(ctypes.byref(d), ctypes.byref(c), x_t.data_ptr(),
                                          B_raw_t.data_ptr(), C_raw_t.data_ptr(), dt_t.data_ptr(),
                                          A.data_ptr(), lam_t.data_ptr(), theta_t.data_ptr(),
                                          ctypes.byref(nc), y_t.data_ptr(), _stream_handle(stream))
    if st != M3_OK:
        raise M3Error(st, "m3_ssm_decode_step_bcnorm")
    return y_t


def m3_ssm_prefill_noalloc(x, B, C, dt, A, lam, theta, h0: State | None = None, *, y,
                           hT: State | None = None, out_dtype=torch.float32, stream=None):
    """m3_ssm_prefill without a workspace, for callers that may not allocate device
    memory: the library's own static device scratch is used instead.  ``y`` must be
    given (this wrapper allocates nothing either).  Every tensor must sit on one device;
    the call runs with that device current, so the scratch of that device is used.
    Calls on one device share that scratch, so calls that overlap on the GPU race;
    order them on one stream."""
    in_dt = x.dtype
    dev = _check_inputs(dict(x=x, B=B, C=C, dt=dt, lam=lam, theta=theta), in_dt)
    _check_inputs(dict(A=A), torch.float32)
    d = _dims(x, dt, theta, 0, in_dt, out_dtype)
    if y.dtype != out_dtype or not y.is_contiguous() or y.numel() != d.B * d.T * d.H * d.R * d.P:
        raise ValueError("y: wrong dtype, layout or size")
    for name, t in (("A", A), ("y", y)):
        if t.device != dev:
            raise ValueError(f"{name}: on {t.device}, inputs on {dev}")
    for name, s in (("h0", h0), ("hT", hT)):
        if s is not None and any(t.device != dev for t in (s.h, s.phi, s.prev_B, s.prev_x)):
            raise ValueError(f"{name}: state tensors must be on {dev}")
    c0 = h0._c() if h0 is not None else None
    c1 = hT._c() if hT is not None else None
    # The library takes the scratch array of the CUDA device that is current during the
    # call, so the call runs with the tensors' device current.
    with torch.cuda.device(dev):
        st = load().m3_ssm_prefill_noalloc(ctypes.byref(d), x.data_ptr(), B.data_ptr(),
                                           C.data_ptr(), dt.data_ptr(), A.data_ptr(),
                                           lam.data_ptr(), theta.data_ptr(),
                                           ctypes.byref(c0) if c0 is not None else None,
                                           y.data_ptr(),
                                           ctypes.byref(c1) if c1 is not None else None,
                                           _stream_handle(stream))
    if st != M3_OK:
        raise M3Error(st, "m3_ssm_prefill_noalloc")
    return y


def m3_ssm_decode_step(state: State, x_t, B_t, C_t, dt_t, A, lam_t, theta_t, *, y_t=None,
                       out_dtype=torch.float32, stream=None):
    """One decode step, updating ``state`` in place.  x_t [B,H,R,P] (or [B,H,P]),
    B_t/C_t [B,H,R,N] (or [B,H,N]), dt_t/lam_t [B,H], theta_t [B,H,N/2].
    Returns y_t [B,H,R,P] in ``out_dtype``."""
    in_dt = x_t.dtype
    dev = _check_inputs(dict(x_t=x_t, B_t=B_t, C_t=C_t, dt_t=dt_t, lam_t=lam_t, theta_t=theta_t),
                        in_dt)
    _check_inputs(dict(A=A), torch.float32)
    d = _dims(x_t, dt_t, theta_t, 0, in_dt, out_dtype, prefill=False)
    if y_t is None:
        y_t = torch.empty(d.B, d.H, d.R, d.P, dtype=out_dtype, device=dev)
    c = state._c()
    st = load().m3_ssm_decode_step(ctypes.byref(d), ctypes.byref(c), x_t.data_ptr(),
                                   B_t.data_ptr(), C_t.data_ptr(), dt_t.data_ptr(), A.data_ptr(),
                                   lam_t.data_ptr(), theta_t.data_ptr(), y_t.data_ptr(),
                                   _stream_handle(stream))
    if st != M3_OK:
        raise M3Error(st, "m3_ssm_decode_step")
    return y_t


def _ssd_dims(x, dt, N, prefill, in_dt, out_dt) -> M3Dims:
    if prefill:
        Bsz, T, H = dt.shape
    else:
        (Bsz, H), T = dt.shape, 0
    return M3Dims(Bsz, T, H, x.shape[-1], N, 1, 0, _DT[in_dt], _DT[out_dt])


def _check_state_h(h, d: M3Dims, dev, what):
    if h is None:
        return None
    if (h.dtype != torch.float32 or not h.is_contiguous() or h.device != dev
            or h.numel() != d.B * d.H * d.N * d.P):
        raise ValueError(f"{what}: float32 [B,H,N,P] contiguous on {dev} expected")
    return h.data_ptr()


def m3_ssd_prefill(x, B, C, dt, A, h0=None, *, y=None, hT=None, workspace=None,
                   out_dtype=torch.float32, stream=None):
    """Mamba-2 special case (lambda = 1, theta = 0) of the prefill, SISO.  x [B,T,H,P],
    B/C [B,T,H,N], dt [B,T,H], A [H] float32; h0 / hT optional float32 [B,H,N,P] states
    (hT may be h0).  Returns y [B,T,H,1,P] in ``out_dtype``."""
    in_dt = x.dtype
    dev = _check_inputs(dict(x=x, B=B, C=C, dt=dt), in_dt)
    _check_inputs(dict(A=A), torch.float32)
    d = _ssd_dims(x, dt, B.shape[-1], True, in_dt, out_dtype)
    if y is None:
        y = torch.empty(d.B, d.T, d.H, 1, d.P, dtype=out_dtype, device=dev)
    elif y.dtype != out_dtype or not y.is_contiguous() or y.numel() != d.B * d.T * d.H * d.P:
        raise ValueError("y: wrong dtype, layout or size")
    if workspace is None:
        workspace = workspace_for(d, dev)
    p0 = _check_state_h(h0, d, dev, "h0")
    p1 = _check_state_h(hT, d, dev, "hT")
    st = load().m3_ssd_prefill(ctypes.byref(d), x.data_ptr(), B.data_ptr(), C.data_ptr(),
                               dt.data_ptr(), A.data_ptr(), p0, y.data_ptr(), p1,
                               workspace.data_ptr(), workspace.numel(), _stream_handle(stream))
    if st != M3_OK:
        raise M3Error(st, "m3_ssd_prefill")
    return y


def m3_ssd_decode_step(h, x_t, B_t, C_t, dt_t, A, *, y_t=None, out_dtype=torch.float32,
                       stream=None):
    """One Mamba-2 decode step, updating the float32 state ``h`` [B,H,N,P] in place.
    x_t [B,H,P], B_t/C_t [B,H,N], dt_t [B,H].  Returns y_t [B,H,1,P] in ``out_dtype``."""
    in_dt = x_t.dtype
    dev = _check_inputs(dict(x_t=x_t, B_t=B_t, C_t=C_t, dt_t=dt_t), in_dt)
    _check_inputs(dict(A=A), torch.float32)
    d = _ssd_dims(x_t, dt_t, B_t.shape[-1], False, in_dt, out_dtype)
    if y_t is None:
        y_t = torch.empty(d.B, d.H, 1, d.P, dtype=out_dtype, device=dev)
    ph = _check_state_h(h, d, dev, "h")
    if ph is None:
        raise ValueError("h: the state is required")
    st = load().m3_ssd_decode_step(ctypes.byref(d), ph, x_t.data_ptr(), B_t.data_ptr(),
                                   C_t.data_ptr(), dt_t.data_ptr(), A.data_ptr(), y_t.data_ptr(),
                                   _stream_handle(stream))
    if st != M3_OK:
        raise M3Error(st, "m3_ssd_decode_step")
    return y_t


def m3_ssm_prefill_backward(x, B, C, dt, A, lam, theta, dy, h0: State | None = None, *,
                            dhT=None, want_dh0=False, workspace=None, stream=None) -> dict:
    """Gradients of L = <dy, y> + <dhT, h_T> for the prefill with these inputs (shapes as
    ``m3_ssm_prefill``; dy like y, in the dtype y had; dhT float32 [B,H,N,P] or None).
    Returns float32 tensors dx, dB, dC, ddt, dA [H], dlambda, dtheta and, if ``want_dh0``,
    dh0 [B,H,N,P]."""
    in_dt = x.dtype
    dev = _check_inputs(dict(x=x, B=B, C=C, dt=dt, lam=lam, theta=theta), in_dt)
    _check_inputs(dict(A=A), torch.float32)
    d = _dims(x, dt, theta, 0, in_dt, dy.dtype)
    _check_inputs(dict(dy=dy), dy.dtype)
    if dy.numel() != d.B * d.T * d.H * d.R * d.P:
        raise ValueError("dy: wrong size")
    if dhT is not None and (dhT.dtype != torch.float32 or not dhT.is_contiguous()
                            or dhT.numel() != d.B * d.H * d.N * d.P):
        raise ValueError("dhT: float32 [B,H,N,P] contiguous expected")
    f32 = dict(dtype=torch.float32, device=dev)
    g = {"dx": torch.empty(d.B, d.T, d.H, d.R, d.P, **f32),
         "dB": torch.empty(d.B, d.T, d.H, d.R, d.N, **f32),
         "dC": torch.empty(d.B, d.T, d.H, d.R, d.N, **f32),
         "ddt": torch.empty(d.B, d.T, d.H, **f32), "dA": torch.empty(d.H, **f32),
         "dlambda": torch.empty(d.B, d.T, d.H, **f32),
         "dtheta": torch.empty(d.B, d.T, d.H, d.N // 2, **f32)}
    if want_dh0:
        g["dh0"] = torch.empty(d.B, d.H, d.N, d.P, **f32)
    if workspace is None:
        n = int(load().m3_ssm_prefill_backward_workspace(ctypes.byref(d)))
        workspace = torch.empty((n + 15) // 16 * 16, dtype=torch.uint8, device=dev)
    c0 = h0._c() if h0 is not None else None
    st = load().m3_ssm_prefill_backward(
        ctypes.byref(d), x.data_ptr(), B.data_ptr(), C.data_ptr(), dt.data_ptr(), A.data_ptr(),
        lam.data_ptr(), theta.data_ptr(), ctypes.byref(c0) if c0 is not None else None,
        dy.data_ptr(), dhT.data_ptr() if dhT is not None else None, g["dx"].data_ptr(),
        g["dB"].data_ptr(), g["dC"].data_ptr(), g["ddt"].data_ptr(), g["dA"].data_ptr(),
        g["dlambda"].data_ptr(), g["dtheta"].data_ptr(),
        g["dh0"].data_ptr() if want_dh0 else None, workspace.data_ptr(), workspace.numel(),
        _stream_handle(stream))
    if st != M3_OK:
        raise M3Error(st, "m3_ssm_prefill_backward")
    return g


def m3_ssm_device_status(workspace: torch.Tensor, stream=None) -> int:
    """Status word of a prefill workspace (waits for the stream): M3_OK or M3_ERR_TIMEOUT."""
    return int(load().m3_ssm_device_status(workspace.data_ptr(), _stream_handle(stream)))
