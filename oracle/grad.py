"""Gradient oracle for the Mamba-3 SSM layer core -- TEST INFRASTRUCTURE ONLY.

Only ``tests/`` and the benchmark's CPU-baseline leg may import this module; the CUDA
path never does, and nothing here touches it.

What it computes: the gradients of the prefill's outputs (y for every token, and the exit
state h_T) with respect to every input, for given output cotangents dy and dh_T -- the
backward pass that training needs ("fast training kernels", paper section 1; the masked
form of section 2.3 / Eq. (7) is the same linear map, so its backward is the transpose of
this recurrence's).

How: the recurrence of ``m3_oracle.c`` is written out once more, token by token, in float64
torch operations (paper notation: Proposition 1 coefficients, Proposition 3 rotation of B
and C by the cumulative angle, the previous token rotated by its own angle (the reading of
Proposition 4 the C oracle takes), MIMO rank-R products of section 3.3), and torch's
reverse-mode autograd differentiates it.  Reverse-mode differentiation of a composition of
elementary operations is the definition of the gradient; there is no blocking or
reordering here.

Pinned, not by re-typing, but by directional finite differences of the C oracle's forward
(tests/test_oracle_grad.py): for random directions v, <grad, v> must match
(L(u + e v) - L(u - e v)) / 2e with L = <dy, y> + <dh_T, h_T> computed by m3_oracle.c.

Small sizes only (pure Python loop over tokens).
"""
from __future__ import annotations

import numpy as np
import torch

INPUTS = ("x", "Bm", "Cm", "dt", "A", "lam", "theta", "h0")


def _rot_t(phi, v):
    """R(phi)^T applied pair by pair: v [..., N] -> (c u + s v, -s u + c v) per pair (2k, 2k+1)."""
    u, w = v[..., 0::2], v[..., 1::2]
    c, s = torch.cos(phi), torch.sin(phi)
    out = torch.stack((c * u + s * w, -s * u + c * w), dim=-1)
    return out.reshape(v.shape)


def forward(x, Bm, Cm, dt, A, lam, theta, h0, phi0, prevB0, prevx0):
    """One sequence.  x [T,R,P]; Bm, Cm [T,R,N]; dt, lam [T]; A scalar; theta [T,N/2];
    h0 [N,P]; phi0 [N/2]; prevB0 [R,N]; prevx0 [R,P].  Returns y [T,R,P], h_T [N,P]."""
    T = x.shape[0]
    h, phi = h0, phi0
    bprev = _rot_t(phi, prevB0)          # B~ of the token before t = 0, by its own angle
    xprev = prevx0
    ys = []
    for t in range(T):
        alpha = torch.exp(dt[t] * A)
        beta = (1 - lam[t]) * dt[t] * alpha
        gamma = lam[t] * dt[t]
        phi = phi + dt[t] * theta[t]
        bt = _rot_t(phi, Bm[t])           # [R, N]
        ct = _rot_t(phi, Cm[t])
        h = alpha * h + beta * (bprev.T @ xprev) + gamma * (bt.T @ x[t])   # [N, P]
        ys.append((h.T @ ct.T).T)         # y_t = h^T C~_t  (P x R), stored [R, P]
        bprev, xprev = bt, x[t]
    return torch.stack(ys), h


def grads(x, Bm, Cm, dt, A, lam, theta, dy, dhT=None, state=None):
    """Gradients of L = <dy, y> + <dhT, h_T> for S sequences.

    Shapes as ``oracle.scan``: x [S,T,R,P]; Bm, Cm [S,T,R,N]; dt, lam [S,T]; A [S];
    theta [S,T,N/2]; dy [S,T,R,P]; dhT [S,N,P] or None; state {h, phi, prev_B, prev_x}
    or None (fresh start).  Returns a dict of float64 numpy arrays with the inputs' shapes:
    x, Bm, Cm, dt, A (per sequence), lam, theta, h0.
    """
    f = lambda a: torch.tensor(np.asarray(a, dtype=np.float64))
    S, T, R, P = np.shape(x)
    N = np.shape(Bm)[-1]
    out = {k: [] for k in INPUTS}
    for i in range(S):
        leaves = {
            "x": f(x[i]), "Bm": f(Bm[i]), "Cm": f(Cm[i]), "dt": f(dt[i]), "A": f(A[i]),
            "lam": f(lam[i]), "theta": f(theta[i]),
            "h0": f(state["h"][i]) if state is not None else torch.zeros(N, P, dtype=torch.float64),
        }
        for v in leaves.values():
            v.requires_grad_(True)
        phi0 = f(state["phi"][i]) if state is not None else torch.zeros(N // 2, dtype=torch.float64)
        pB = f(state["prev_B"][i]) if state is not None else torch.zeros(R, N, dtype=torch.float64)
        px = f(state["prev_x"][i]) if state is not None else torch.zeros(R, P, dtype=torch.float64)
        y, hT = forward(leaves["x"], leaves["Bm"], leaves["Cm"], leaves["dt"], leaves["A"],
                        leaves["lam"], leaves["theta"], leaves["h0"], phi0, pB, px)
        loss = (y * f(dy[i])).sum()
        if dhT is not None:
            loss = loss + (hT * f(dhT[i])).sum()
        g = torch.autograd.grad(loss, [leaves[k] for k in INPUTS], allow_unused=True)
        for k, gk in zip(INPUTS, g):
            out[k].append(np.zeros(leaves[k].shape) if gk is None else gk.detach().numpy())
    return {k: np.stack(v) for k, v in out.items()}
