"""Pins of the fp64 oracle against facts the paper fixes, independent of the oracle's own code.

Each test rebuilds the expected result by a different route: a hand-worked
example, a closed form, a special case that reduces to a textbook rule, an
equivalent formulation of the method (explicit complex state, explicit T x T
masked matrix), or an invariant (continuation, linearity).  A plausible slip
in the oracle -- a dropped beta term, a wrong rotation sign, the wrong angle
on the previous-token term, a transposed MIMO operand -- fails at least one.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_seq(rng, S, T, N, P, R, lam=None, theta_scale=1.0):
    x = rng.standard_normal((S, T, R, P))
    Bm = rng.standard_normal((S, T, R, N)) / np.sqrt(N * R)
    Cm = rng.standard_normal((S, T, R, N)) / np.sqrt(N * R)
    dt = np.log1p(np.exp(rng.normal(-2, 0.5, (S, T))))
    A = -np.exp(rng.uniform(0, np.log(16), S))
    lam = 1 / (1 + np.exp(-rng.standard_normal((S, T)))) if lam is None else np.full((S, T), lam)
    theta = theta_scale * rng.standard_normal((S, T, N // 2))
    return dict(x=x, Bm=Bm, Cm=Cm, dt=dt, A=A, lam=lam, theta=theta)


def rand_state(rng, S, N, P, R):
    return {
        "h": rng.standard_normal((S, N, P)),
        "phi": rng.uniform(-7, 7, (S, N // 2)),
        "prev_B": rng.standard_normal((S, R, N)) / np.sqrt(N * R),
        "prev_x": rng.standard_normal((S, R, P)),
    }


def rot_t(phi, v):
    """R(phi)^T applied pair-wise along the last axis (pairs (2k, 2k+1))."""
    c, s = np.cos(phi), np.sin(phi)
    u, w = v[..., 0::2], v[..., 1::2]
    out = np.empty_like(v)
    out[..., 0::2] = c * u + s * w
    out[..., 1::2] = -s * u + c * w
    return out


# ---------------------------------------------------------------- golden examples


def test_hand_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "hand_example.json")))
    i = g["inputs"]
    T = i["T"]
    x = np.array(i["x"], float).reshape(1, T, 1, 1)
    Bm = np.array(i["B"], float).reshape(1, T, 1, 2)
    Cm = np.array(i["C"], float).reshape(1, T, 1, 2)
    y, st, _ = oracle.scan(x, Bm, Cm, np.array([i["dt"]]), [i["A"]], np.array([i["lambda"]]),
                           np.array(i["theta_pair0"]).reshape(1, T, 1))
    e = g["expected"]
    np.testing.assert_allclose(y.ravel(), e["y"], atol=1e-14)
    np.testing.assert_allclose(st["h"].ravel(), e["h_final"], atol=1e-14)
    np.testing.assert_allclose(st["phi"].ravel(), e["phi_final"], atol=1e-14)
    np.testing.assert_allclose(st["prev_B"].ravel(), e["prev_B_final"], atol=0)
    np.testing.assert_allclose(st["prev_x"].ravel(), e["prev_x_final"], atol=0)


def test_parity_construction():
    """(e) Paper section 3.2: a rotation by pi per 1-bit tracks parity exactly."""
    g = json.load(open(os.path.join(GOLDEN, "parity_example.json")))
    bits = np.array(g["bits"], float)
    T, N = len(bits), 4
    x = np.zeros((1, T, 1, 1))
    x[0, 0] = 1.0
    Bm = np.zeros((1, T, 1, N))
    Bm[..., 0] = 1.0
    theta = np.zeros((1, T, N // 2))
    theta[0, :, 0] = np.pi * bits
    theta[0, :, 1] = 0.37  # a second pair that carries no signal must not leak into y
    y, _, _ = oracle.scan(x, Bm, Bm.copy(), np.ones((1, T)), [0.0], np.ones((1, T)), theta)
    np.testing.assert_allclose(y.ravel(), g["expected_y"], atol=1e-12)


# ---------------------------------------------------------------- special cases


@pytest.mark.parametrize("R", [1, 3])
def test_lambda_one_theta_zero_is_exponential_euler(R):
    """(a) lambda = 1, theta = 0: the Mamba-2 exponential-Euler rule h = e^{dt A} h + dt B X^T
    (paper Eq. 4; aipaper.cc summary: 'when lambda = 1 the formula reduces to Mamba-2')."""
    rng = np.random.default_rng(1)
    S, T, N, P = 2, 40, 6, 5
    d = rand_seq(rng, S, T, N, P, R, lam=1.0, theta_scale=0.0)
    y, st, _ = oracle.scan(**d)
    for s in range(S):
        h = np.zeros((N, P))
        for t in range(T):
            Bt = d["Bm"][s, t].T  # N x R
            Xt = d["x"][s, t].T  # P x R
            h = np.exp(d["dt"][s, t] * d["A"][s]) * h + d["dt"][s, t] * Bt @ Xt.T
            yt = h.T @ d["Cm"][s, t].T  # P x R
            np.testing.assert_allclose(y[s, t].T, yt, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(st["h"][s], h, rtol=1e-12, atol=1e-12)


def test_explicit_complex_state_equals_absorbed_rope():
    """(b) Propositions 2-4: the complex state, evolved explicitly with transition
    exp(dt (A + i theta)) on each pair, gives the same y as the RoPE-absorbed real form.
    Left trapezoid endpoint: (1 - lambda) dt exp(dt (A + i theta)) b_{t-1} x_{t-1}."""
    rng = np.random.default_rng(2)
    S, T, N, P, R = 2, 50, 8, 3, 2
    d = rand_seq(rng, S, T, N, P, R)
    st0 = rand_state(rng, S, N, P, R)
    y, st, _ = oracle.scan(**d, state=st0)
    K = N // 2
    for s in range(S):
        # complex state z[k, p]; real pair (2k, 2k+1) <-> Re, Im.  The explicit frame is the
        # absorbed frame rotated back by the entry angle: h^e = R(phi) h.
        h0 = st0["h"][s]
        phi = st0["phi"][s]
        z = np.exp(1j * phi)[:, None] * (h0[0::2] + 1j * h0[1::2])
        pb = st0["prev_B"][s]  # R x N, raw previous token
        bprev = pb[:, 0::2] + 1j * pb[:, 1::2]  # R x K
        xprev = st0["prev_x"][s]  # R x P
        for t in range(T):
            dt, lam = d["dt"][s, t], d["lam"][s, t]
            mu = (dt * (d["A"][s] + 1j * d["theta"][s, t]))[:, None]  # K x 1
            b = d["Bm"][s, t][:, 0::2] + 1j * d["Bm"][s, t][:, 1::2]
            c = d["Cm"][s, t][:, 0::2] + 1j * d["Cm"][s, t][:, 1::2]
            xt = d["x"][s, t]
            z = (np.exp(mu) * z + (1 - lam) * dt * np.exp(mu) * (bprev.T @ xprev)
                 + lam * dt * (b.T @ xt))
            # y[p, r] = sum_k Re(conj(c_k) z_k) = C^T h^e
            yt = np.real(np.conj(c) @ z)  # R x P
            np.testing.assert_allclose(y[s, t], yt, rtol=1e-10, atol=1e-11)
            bprev, xprev = b, xt
        phiT = st["phi"][s]
        he = np.empty((N, P))
        he[0::2], he[1::2] = z.real, z.imag
        np.testing.assert_allclose(_rot_t_rows(phiT, he), st["h"][s], rtol=1e-10, atol=1e-11)


def _rot_t_rows(phi, h):
    """R(phi_k)^T applied to row pairs (2k, 2k+1) of an N x P matrix."""
    c, s = np.cos(phi)[:, None], np.sin(phi)[:, None]
    out = np.empty_like(h)
    out[0::2] = c * h[0::2] + s * h[1::2]
    out[1::2] = -s * h[0::2] + c * h[1::2]
    return out


@pytest.mark.parametrize("R", [1, 3])
def test_recurrence_equals_bruteforce_masked_form(R):
    """(c) Section 2.3 / Eq. (7): y = ((L . Bd) o (C~ B~^T)) X plus the entry-state terms, where
    L is the 1-semiseparable decay mask, L[t,s] = prod_{k=s+1..t} alpha_k, and Bd the 2-band
    convolution matrix (diagonal gamma_s, sub-diagonal beta_s).  For MIMO the mask is
    expanded by J_R (all rank pairs of one token pair interact)."""
    rng = np.random.default_rng(3)
    S, T, N, P = 2, 48, 6, 4
    d = rand_seq(rng, S, T, N, P, R)
    st0 = rand_state(rng, S, N, P, R)
    y, st, _ = oracle.scan(**d, state=st0)
    for s in range(S):
        dt, lam, A = d["dt"][s], d["lam"][s], d["A"][s]
        alpha = np.exp(dt * A)
        beta = (1 - lam) * dt * alpha
        gamma = lam * dt
        L = np.zeros((T, T))
        for t in range(T):
            for u in range(t + 1):
                L[t, u] = np.prod(alpha[u + 1:t + 1])
        Bd = np.diag(gamma) + np.diag(beta[1:], -1)
        M = L @ Bd
        phi = st0["phi"][s][None, :] + np.cumsum(dt[:, None] * d["theta"][s], axis=0)  # T x K
        Bt = rot_t(phi[:, None, :], d["Bm"][s])  # T x R x N
        Ct = rot_t(phi[:, None, :], d["Cm"][s])
        Bp = rot_t(st0["phi"][s][None, :], st0["prev_B"][s])  # R x N, rotated by entry angle
        rows_C = Ct.reshape(T * R, N)
        rows_B = Bt.reshape(T * R, N)
        X = d["x"][s].reshape(T * R, P)
        Mx = np.kron(M, np.ones((R, R)))
        Y = (Mx * (rows_C @ rows_B.T)) @ X
        # entry state: prod_{k<=t} alpha_k C~_t h0, and the first token's beta term
        # beta_0 * L[t, 0] * C~_t B~_{-1} X_{-1}^T.
        decay = np.cumprod(alpha)
        Y += (decay[:, None, None] * (Ct @ st0["h"][s])).reshape(T * R, P)
        v_prev = Bp.T @ st0["prev_x"][s]  # N x P
        Y += ((beta[0] * L[:, 0])[:, None, None] * (Ct @ v_prev)).reshape(T * R, P)
        np.testing.assert_allclose(y[s].reshape(T * R, P), Y, rtol=1e-10, atol=1e-11)


def test_mimo_is_sum_of_siso_runs():
    """(d) Section 3.3: with shared dt, lambda, theta, the rank-R state is the sum over input
    columns r of SISO states driven by (B[:, r], X[:, r]); output column r' reads it with
    C[:, r'].  So MIMO y[:, r'] = sum_r SISO(x_r, B_r, C_r') -- and R = 1 is SISO itself."""
    rng = np.random.default_rng(4)
    S, T, N, P, R = 2, 30, 6, 4, 3
    d = rand_seq(rng, S, T, N, P, R)
    y, st, _ = oracle.scan(**d)
    ysum = np.zeros_like(y)
    hsum = np.zeros_like(st["h"])
    for r in range(R):
        for rp in range(R):
            dd = dict(d)
            dd["x"] = d["x"][:, :, r:r + 1]
            dd["Bm"] = d["Bm"][:, :, r:r + 1]
            dd["Cm"] = d["Cm"][:, :, rp:rp + 1]
            y1, st1, _ = oracle.scan(**dd)
            ysum[:, :, rp] += y1[:, :, 0]
            if rp == 0:
                hsum += st1["h"]
    np.testing.assert_allclose(y, ysum, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(st["h"], hsum, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- accuracy order


def _ode_run(dt_step, lam, A, omega_rot, nu, t_end=1.0):
    """Oracle on one rotation pair with constant dt, A, theta and input x(s) = sin(nu s)."""
    T = int(round(t_end / dt_step)) + 1
    s = np.arange(T) * dt_step
    R, N, P = 2, 2, 1
    x = np.zeros((1, T, R, P))
    x[0, :, 0, 0] = np.sin(nu * s)
    Bm = np.zeros((1, T, R, N))
    Bm[0, :, 0, 0] = 1.0  # b = 1 (real input on the first component)
    Cm = np.zeros((1, T, R, N))
    Cm[0, :, 0, 0] = 1.0  # read Re z
    Cm[0, :, 1, 1] = 1.0  # read Im z
    theta = np.full((1, T, 1), omega_rot)
    y, _, _ = oracle.scan(x, Bm, Cm, np.full((1, T), dt_step), [A], np.full((1, T), lam), theta)
    return y[0, -1, :, 0]  # (Re z, Im z) at s = t_end


def _closed_form(A, omega_rot, nu, s):
    mu = A + 1j * omega_rot
    return (-mu * np.sin(nu * s) - nu * np.cos(nu * s) + nu * np.exp(mu * s)) / (mu * mu + nu * nu)


@pytest.mark.parametrize("lam,order", [(0.5, 2), (1.0, 1)])
def test_trapezoid_is_second_order_euler_first(lam, order):
    """(f1) Section 3.1: the exponential-trapezoid (lambda = 1/2) has global error O(dt^2); the
    exponential-Euler rule (lambda = 1) O(dt).  Closed form of h' = A h + sin(nu s), h(0) = 0."""
    A, nu = -1.0, 3.0
    exact = _closed_form(A, 0.0, nu, 1.0).real
    errs = [abs(_ode_run(h, lam, A, 0.0, nu)[0] - exact) for h in (0.02, 0.01, 0.005)]
    ratios = [errs[0] / errs[1], errs[1] / errs[2]]
    for r in ratios:
        assert abs(np.log2(r) - order) < 0.15, (errs, ratios)


def test_complex_pair_matches_analytic_rotation():
    """(f2) Sections 3.2.1-3.2.2: one complex eigenvalue A + i theta; the discrete output
    converges at second order to z' = (A + i theta) z + sin(nu s).  A wrong rotation sign, or
    the previous-token term rotated by the current angle instead of its own, breaks this."""
    A, om, nu = -0.7, 5.0, 2.0
    exact = _closed_form(A, om, nu, 1.0)
    errs = []
    for h in (0.02, 0.01, 0.005):
        re, im = _ode_run(h, 0.5, A, om, nu)
        errs.append(abs(re + 1j * im - exact))
    assert errs[-1] < 1e-4
    for a, b in zip(errs, errs[1:]):
        assert abs(np.log2(a / b) - 2) < 0.15, errs


# ---------------------------------------------------------------- invariants


def test_continuation_across_calls():
    """(g) The state (h, phi, previous token) carries a sequence across calls exactly."""
    rng = np.random.default_rng(5)
    S, T, N, P, R = 2, 64, 8, 4, 2
    d = rand_seq(rng, S, T, N, P, R)
    st0 = rand_state(rng, S, N, P, R)
    y, st, _ = oracle.scan(**d, state=st0)
    for T1 in (1, 17, 63):
        a = {k: (v[:, :T1] if v.ndim >= 2 and k != "A" else v) for k, v in d.items()}
        b = {k: (v[:, T1:] if v.ndim >= 2 and k != "A" else v) for k, v in d.items()}
        y1, s1, _ = oracle.scan(**a, state=st0)
        y2, s2, _ = oracle.scan(**b, state=s1)
        np.testing.assert_array_equal(np.concatenate([y1, y2], 1), y)
        for k in st:
            np.testing.assert_array_equal(s2[k], st[k])


def test_linearity_in_inputs_and_state():
    """(h) For fixed B, C, dt, lambda, theta and previous B, the map (x, h0, prev_x) -> (y, h_T)
    is linear (the system is a linear time-varying SSM, paper section 3.1)."""
    rng = np.random.default_rng(6)
    S, T, N, P, R = 1, 40, 6, 3, 2
    d = rand_seq(rng, S, T, N, P, R)
    s1, s2 = rand_state(rng, S, N, P, R), rand_state(rng, S, N, P, R)
    s2["phi"], s2["prev_B"] = s1["phi"], s1["prev_B"]
    x1, x2 = d["x"], rng.standard_normal(d["x"].shape)
    a, b = 0.7, -1.3
    ya, sa, _ = oracle.scan(**{**d, "x": x1}, state=s1)
    yb, sb, _ = oracle.scan(**{**d, "x": x2}, state=s2)
    sc = dict(s1)
    sc["h"] = a * s1["h"] + b * s2["h"]
    sc["prev_x"] = a * s1["prev_x"] + b * s2["prev_x"]
    yc, scc, _ = oracle.scan(**{**d, "x": a * x1 + b * x2}, state=sc)
    np.testing.assert_allclose(yc, a * ya + b * yb, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(scc["h"], a * sa["h"] + b * sb["h"], rtol=1e-10, atol=1e-11)


def test_batch_threads_agree():
    """Spreading sequences over threads changes nothing (each sequence is independent)."""
    rng = np.random.default_rng(7)
    d = rand_seq(rng, 5, 20, 4, 3, 2)
    y1, s1, _ = oracle.scan(**d, nthreads=1)
    y4, s4, _ = oracle.scan(**d, nthreads=4)
    np.testing.assert_array_equal(y1, y4)
    np.testing.assert_array_equal(s1["h"], s4["h"])
