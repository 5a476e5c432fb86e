"""The finite-difference pin of the gradient oracle catches plausible mistakes.

Each mutation below is planted in a copy of oracle/grad.py's forward (the function it
differentiates); the gradients it then produces must disagree with central finite differences
of the C oracle for at least one input.  This checks the pin, not the oracle."""
import numpy as np
import pytest
import torch

from oracle import grad as G
from tests.test_oracle_grad import loss_c, problem


def mutated_forward(kind):
    def fwd(x, Bm, Cm, dt, A, lam, theta, h0, phi0, prevB0, prevx0):
        T = x.shape[0]
        h, phi = h0, phi0
        bprev = G._rot_t(phi, prevB0)
        xprev = prevx0
        ys = []
        for t in range(T):
            alpha = torch.exp(dt[t] * A)
            beta = (1 - lam[t]) * dt[t] * (1.0 if kind == "beta_without_alpha" else alpha)
            gamma = lam[t] * (1.0 if kind == "gamma_without_dt" else dt[t])
            phi_new = phi + dt[t] * theta[t]
            bt = G._rot_t(phi_new, Bm[t])
            ct = G._rot_t(-phi_new if kind == "c_rotated_the_other_way" else phi_new, Cm[t])
            if kind == "prev_token_at_new_angle":
                bprev = G._rot_t(phi_new, Bm[t - 1]) if t > 0 else G._rot_t(phi_new, prevB0)
            h = alpha * h + beta * (bprev.T @ xprev) + gamma * (bt.T @ x[t])
            ys.append((h.T @ ct.T).T)
            bprev, xprev = bt, x[t]
            phi = phi_new
        return torch.stack(ys), h
    return fwd


@pytest.mark.parametrize("kind", ["beta_without_alpha", "gamma_without_dt",
                                  "c_rotated_the_other_way", "prev_token_at_new_angle"])
def test_each_mutation_fails_the_finite_difference_pin(kind, monkeypatch):
    S, T, N, P, R = 2, 6, 4, 3, 2
    u, state, dy, dhT, rng = problem(S, T, N, P, R, 21, False)
    monkeypatch.setattr(G, "forward", mutated_forward(kind))
    g = G.grads(u["x"], u["Bm"], u["Cm"], u["dt"], u["A"], u["lam"], u["theta"], dy, dhT, state)
    eps, worst = 1e-6, 0.0
    for name in u:
        v = rng.standard_normal(np.shape(u[name]))
        up, um = dict(u), dict(u)
        up[name] = u[name] + eps * v
        um[name] = u[name] - eps * v
        fd = (loss_c(up, state, dy, dhT) - loss_c(um, state, dy, dhT)) / (2 * eps)
        gv = float(np.sum(g[name] * v))
        worst = max(worst, abs(gv - fd) / max(1.0, abs(fd)))
    assert worst > 1e-3, (kind, worst)


def test_the_unmutated_copy_passes(monkeypatch):
    """Control: the copy above without a mutation agrees with the finite differences, so the
    failures come from the planted mistakes."""
    S, T, N, P, R = 2, 6, 4, 3, 2
    u, state, dy, dhT, rng = problem(S, T, N, P, R, 21, False)
    monkeypatch.setattr(G, "forward", mutated_forward("none"))
    g = G.grads(u["x"], u["Bm"], u["Cm"], u["dt"], u["A"], u["lam"], u["theta"], dy, dhT, state)
    eps = 1e-6
    for name in u:
        v = rng.standard_normal(np.shape(u[name]))
        up, um = dict(u), dict(u)
        up[name] = u[name] + eps * v
        um[name] = u[name] - eps * v
        fd = (loss_c(up, state, dy, dhT) - loss_c(um, state, dy, dhT)) / (2 * eps)
        assert abs(float(np.sum(g[name] * v)) - fd) <= 1e-6 * max(1.0, abs(fd)), name
