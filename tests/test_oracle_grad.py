"""Pins of the gradient oracle (oracle/grad.py) against the C oracle's forward.

For every input u and random directions v, the oracle's gradient must give the directional
derivative of L = <dy, y> + <dh_T, h_T>, where y and h_T come from m3_oracle.c (code the
gradient oracle does not share), by central differences in float64.  A dropped term, a wrong
sign or a transposed operand anywhere in the backward changes some directional derivative by
O(1) and fails here.  Also: the gradient oracle's own forward equals the C oracle's.
"""
import numpy as np
import pytest

import oracle
from oracle import grad as G


def problem(S, T, N, P, R, seed, fresh):
    rng = np.random.Generator(np.random.PCG64(seed))
    u = {
        "x": rng.standard_normal((S, T, R, P)),
        "Bm": rng.standard_normal((S, T, R, N)) / np.sqrt(N),
        "Cm": rng.standard_normal((S, T, R, N)) / np.sqrt(N),
        "dt": rng.uniform(0.05, 0.6, (S, T)),
        "A": -rng.uniform(0.5, 3.0, S),
        "lam": rng.uniform(0.0, 1.0, (S, T)),
        "theta": rng.standard_normal((S, T, N // 2)),
    }
    state = None if fresh else {
        "h": rng.standard_normal((S, N, P)),
        "phi": rng.uniform(-3, 3, (S, N // 2)),
        "prev_B": rng.standard_normal((S, R, N)) / np.sqrt(N),
        "prev_x": rng.standard_normal((S, R, P)),
    }
    dy = rng.standard_normal((S, T, R, P))
    dhT = rng.standard_normal((S, N, P))
    return u, state, dy, dhT, rng


def loss_c(u, state, dy, dhT, h0=None):
    st = None
    if state is not None or h0 is not None:
        st = dict(state) if state is not None else oracle.zero_state(*np.shape(u["x"])[:1],
                                                                       np.shape(u["Bm"])[-1],
                                                                       np.shape(u["x"])[-1],
                                                                       np.shape(u["x"])[2])
        if h0 is not None:
            st["h"] = h0
    y, sT, _ = oracle.scan(u["x"], u["Bm"], u["Cm"], u["dt"], u["A"], u["lam"], u["theta"], st)
    return float(np.sum(y * dy) + np.sum(sT["h"] * dhT))


@pytest.mark.parametrize("R", [1, 2])
@pytest.mark.parametrize("fresh", [True, False])
def test_gradients_match_finite_differences_of_the_c_oracle(R, fresh):
    S, T, N, P = 2, 7, 4, 3
    u, state, dy, dhT, rng = problem(S, T, N, P, R, 11 + R + 2 * fresh, fresh)
    g = G.grads(u["x"], u["Bm"], u["Cm"], u["dt"], u["A"], u["lam"], u["theta"], dy, dhT, state)
    eps = 1e-6
    names = list(u) + ["h0"]
    for name in names:
        for _ in range(3):
            if name == "h0":
                base = state["h"] if state is not None else np.zeros((S, N, P))
                v = rng.standard_normal(base.shape)
                lp = loss_c(u, state, dy, dhT, h0=base + eps * v)
                lm = loss_c(u, state, dy, dhT, h0=base - eps * v)
                gv = float(np.sum(g["h0"] * v))
            else:
                v = rng.standard_normal(np.shape(u[name]))
                up, um = dict(u), dict(u)
                up[name] = u[name] + eps * v
                um[name] = u[name] - eps * v
                lp, lm = loss_c(up, state, dy, dhT), loss_c(um, state, dy, dhT)
                gv = float(np.sum(g[name] * v))
            fd = (lp - lm) / (2 * eps)
            assert abs(gv - fd) <= 1e-6 * max(1.0, abs(fd)), (name, gv, fd)


def test_gradient_oracle_forward_equals_c_oracle():
    import torch
    S, T, N, P, R = 2, 9, 6, 4, 2
    u, state, dy, dhT, _ = problem(S, T, N, P, R, 5, False)
    yc, sc, _ = oracle.scan(u["x"], u["Bm"], u["Cm"], u["dt"], u["A"], u["lam"], u["theta"], state)
    f = lambda a: torch.tensor(np.asarray(a, dtype=np.float64))
    for i in range(S):
        y, hT = G.forward(f(u["x"][i]), f(u["Bm"][i]), f(u["Cm"][i]), f(u["dt"][i]), f(u["A"][i]),
                          f(u["lam"][i]), f(u["theta"][i]), f(state["h"][i]), f(state["phi"][i]),
                          f(state["prev_B"][i]), f(state["prev_x"][i]))
        np.testing.assert_allclose(y.numpy(), yc[i], rtol=0, atol=1e-12)
        np.testing.assert_allclose(hT.numpy(), sc["h"][i], rtol=0, atol=1e-12)


def test_gradient_of_a_single_token_closed_form():
    """T = 1, fresh start, R = 1: y = gamma (C~ . B~) x with C~ . B~ = C . B (one rotation
    applied to both), so dL/dx = gamma (C . B) dy and dL/dlambda = dt (C . B) <x, dy>."""
    rng = np.random.Generator(np.random.PCG64(3))
    N, P = 6, 5
    x = rng.standard_normal((1, 1, 1, P))
    Bm, Cm = rng.standard_normal((1, 1, 1, N)), rng.standard_normal((1, 1, 1, N))
    dt, lam = np.array([[0.3]]), np.array([[0.7]])
    theta = rng.standard_normal((1, 1, N // 2))
    dy = rng.standard_normal((1, 1, 1, P))
    g = G.grads(x, Bm, Cm, dt, np.array([-1.0]), lam, theta, dy)
    cb = float(Cm[0, 0, 0] @ Bm[0, 0, 0])
    np.testing.assert_allclose(g["x"][0, 0, 0], 0.7 * 0.3 * cb * dy[0, 0, 0], rtol=1e-12)
    np.testing.assert_allclose(g["lam"][0, 0], 0.3 * cb * float(x[0, 0, 0] @ dy[0, 0, 0]), rtol=1e-12)
    np.testing.assert_allclose(g["theta"], 0.0, atol=1e-12)  # the rotation cancels in C . B
    np.testing.assert_allclose(g["A"], 0.0, atol=1e-12)      # h starts at 0: alpha multiplies 0
