"""The chunked (masked-form) adjoint a tensor-core backward pass computes equals the gradient
oracle.  The forward's chunked form is pinned against the recurrence in test_oracle_pins
(brute-force masked form); this pins the backward's: per chunk, with the local natural-log
decay sums ell, the weights w_s = gamma_s + q_{s+1} (q = (1 - lambda) dt), the mask
Mh[i,s] = exp(ell_i - ell_s) w_s below the diagonal and gamma_i on it, and the folded entry
state H_in' = H_in + q_0 B~_{-1}^T X_{-1}:
   h_i = exp(ell_i) H_in' + sum_{s<=i} Mh[i,s] B~_s^T X_s,  Y_i = C~_i h_i;
and backwards, with Gh_i = C~_i^T dY_i plus the exit cotangent at the last token:
   dC~_i = exp(ell_i) dY_i H_in'^T + sum_s D[i,s] B~_s,  D[i,s] = Mh[i,s] dY_i X_s^T,
   dB~_s = sum_i D[i,s]^T C~_i + Mh[last,s] X_s G_out^T,
   dX_s = sum_i Mh[i,s] (C~_i B~_s^T)^T dY_i + Mh[last,s] B~_s G_out,
   dH_in' = sum_i exp(ell_i) Gh_i,
   dMh[i,s] = sum (C~_i B~_s^T) o (dY_i X_s^T) (+ <G_out, B~_s^T X_s> on the last row),
then the chain rule through ell, w, gamma, q, the fold and the rotation (reverse cumulative
sum of d phi over the sequence).  Written here with explicit loops; compared to 1e-9.
"""
import numpy as np
import pytest

from oracle import grad as G


def rot_t(c, s, v):
    out = np.empty_like(v)
    out[..., 0::2] = c * v[..., 0::2] + s * v[..., 1::2]
    out[..., 1::2] = -s * v[..., 0::2] + c * v[..., 1::2]
    return out


def backward_chunked(x, Bm, Cm, dt, A, lam, theta, dy, dhT, h0, phi0, pB0, px0, c):
    T, R, P = x.shape
    N = Bm.shape[-1]
    K = N // 2
    # per-token quantities
    phi = np.empty((T, K)); p = phi0.copy()
    for t in range(T):
        p = p + dt[t] * theta[t]; phi[t] = p
    cs, sn = np.cos(phi), np.sin(phi)
    Bt = rot_t(cs[:, None, :], sn[:, None, :], Bm)   # [T,R,N]
    Ct = rot_t(cs[:, None, :], sn[:, None, :], Cm)
    Bprev0 = rot_t(np.cos(phi0), np.sin(phi0), pB0)   # [R,N]
    q = (1 - lam) * dt
    gam = lam * dt
    a = dt * A                                         # log alpha
    nch = (T + c - 1) // c
    # forward: chunk entry states
    Hin = [None] * nch
    H = h0.copy()
    for k in range(nch):
        t0, t1 = k * c, min(T, (k + 1) * c)
        Hin[k] = H.copy()
        bp, xp = (Bprev0, px0) if t0 == 0 else (Bt[t0 - 1], x[t0 - 1])
        Hp = H + q[t0] * bp.T @ xp
        ell = np.cumsum(a[t0:t1])
        n = t1 - t0
        hs = []
        for i in range(n):
            h = np.exp(ell[i]) * Hp
            for s_ in range(i + 1):
                m = gam[t0 + i] if s_ == i else np.exp(ell[i] - ell[s_]) * (gam[t0 + s_] + q[t0 + s_ + 1])
                h = h + m * Bt[t0 + s_].T @ x[t0 + s_]
            hs.append(h)
        H = hs[-1]
    # backward
    dBt = np.zeros_like(Bt); dCt = np.zeros_like(Ct); dX = np.zeros_like(x)
    dq = np.zeros(T); dgam = np.zeros(T); da = np.zeros(T)
    Gout = dhT.copy()
    for k in reversed(range(nch)):
        t0, t1 = k * c, min(T, (k + 1) * c)
        n = t1 - t0
        bp, xp = (Bprev0, px0) if t0 == 0 else (Bt[t0 - 1], x[t0 - 1])
        Hp = Hin[k] + q[t0] * bp.T @ xp
        ell = np.cumsum(a[t0:t1])
        Mh = np.zeros((n, n))
        for i in range(n):
            for s_ in range(i + 1):
                Mh[i, s_] = gam[t0 + i] if s_ == i else np.exp(ell[i] - ell[s_]) * (gam[t0 + s_] + q[t0 + s_ + 1])
        Cc, Bc, Xc, dYc = Ct[t0:t1], Bt[t0:t1], x[t0:t1], dy[t0:t1]
        # Gh_i = C~_i^T dY_i (+ G_out at the last token)
        Gh = np.einsum("irn,irp->inp", Cc, dYc)
        Gh[n - 1] += Gout
        # gradient contributions
        dHp = np.einsum("i,inp->np", np.exp(ell), Gh)
        dexp = np.einsum("inp,np->i", Gh, Hp)                      # d exp(ell_i)
        dCt[t0:t1] += np.exp(ell)[:, None, None] * np.einsum("irp,np->irn", dYc, Hp)
        dM = np.zeros((n, n))
        for i in range(n):
            for s_ in range(i + 1):
                D = Mh[i, s_] * dYc[i] @ Xc[s_].T                    # R x R
                dCt[t0 + i] += D @ Bc[s_]
                dBt[t0 + s_] += D.T @ Cc[i]
                dX[t0 + s_] += Mh[i, s_] * (Cc[i] @ Bc[s_].T).T @ dYc[i]
                dM[i, s_] += np.sum((Cc[i] @ Bc[s_].T) * (dYc[i] @ Xc[s_].T))
        for s_ in range(n):   # the exit-state cotangent through the last row of the mask
            dBt[t0 + s_] += Mh[n - 1, s_] * Xc[s_] @ Gout.T
            dX[t0 + s_] += Mh[n - 1, s_] * Bc[s_] @ Gout
            dM[n - 1, s_] += np.sum(Gout * (Bc[s_].T @ Xc[s_]))
        # mask parameters -> ell, gamma, w
        dell = dexp * np.exp(ell)
        for i in range(n):
            for s_ in range(i):
                e = np.exp(ell[i] - ell[s_])
                w = gam[t0 + s_] + q[t0 + s_ + 1]
                g = dM[i, s_] * e * w
                dell[i] += g
                dell[s_] -= g
                dgam[t0 + s_] += dM[i, s_] * e
                dq[t0 + s_ + 1] += dM[i, s_] * e
            dgam[t0 + i] += dM[i, i]
        # ell_i = sum_{s <= i} a_s within the chunk
        da[t0:t1] += np.cumsum(dell[::-1])[::-1]
        # the fold H_in' = H_in + q_{t0} B~_{t0-1}^T X_{t0-1}
        dq[t0] += np.sum(dHp * (bp.T @ xp))
        if t0 > 0:
            dBt[t0 - 1] += q[t0] * xp @ dHp.T
            dX[t0 - 1] += q[t0] * bp @ dHp
        Gout = dHp
    dh0 = Gout
    # rotation adjoint and the reverse cumulative sum of d phi
    dB = np.empty_like(Bm); dC = np.empty_like(Cm)
    dB[..., 0::2] = cs[:, None] * dBt[..., 0::2] - sn[:, None] * dBt[..., 1::2]
    dB[..., 1::2] = sn[:, None] * dBt[..., 0::2] + cs[:, None] * dBt[..., 1::2]
    dC[..., 0::2] = cs[:, None] * dCt[..., 0::2] - sn[:, None] * dCt[..., 1::2]
    dC[..., 1::2] = sn[:, None] * dCt[..., 0::2] + cs[:, None] * dCt[..., 1::2]
    dphi = np.sum(dBt[..., 0::2] * Bt[..., 1::2] - dBt[..., 1::2] * Bt[..., 0::2]
                  + dCt[..., 0::2] * Ct[..., 1::2] - dCt[..., 1::2] * Ct[..., 0::2], axis=1)   # [T,K]
    Gphi = np.cumsum(dphi[::-1], axis=0)[::-1]
    dtheta = dt[:, None] * Gphi
    ddt = np.sum(theta * Gphi, axis=1) + da * A + lam * dgam + (1 - lam) * dq
    dlam = dt * (dgam - dq)
    dA = float(np.sum(da * dt))
    return dict(x=dX, Bm=dB, Cm=dC, dt=ddt, lam=dlam, theta=dtheta, A=dA, h0=dh0)




@pytest.mark.parametrize("T,N,P,R,c,fresh", [(7, 4, 3, 1, 3, True), (11, 6, 5, 2, 4, False),
                                            (9, 4, 2, 4, 2, False), (12, 8, 4, 1, 12, False),
                                            (5, 4, 3, 2, 1, False)])
def test_chunked_adjoint_equals_gradient_oracle(T, N, P, R, c, fresh):
    rng = np.random.Generator(np.random.PCG64(T * 100 + N * 10 + R))
    S = 2
    x = rng.standard_normal((S, T, R, P))
    Bm = rng.standard_normal((S, T, R, N)) / np.sqrt(N)
    Cm = rng.standard_normal((S, T, R, N)) / np.sqrt(N)
    dt = rng.uniform(0.05, 0.6, (S, T))
    A = -rng.uniform(0.5, 3, S)
    lam = rng.uniform(0, 1, (S, T))
    theta = rng.standard_normal((S, T, N // 2))
    dy = rng.standard_normal((S, T, R, P))
    dhT = rng.standard_normal((S, N, P))
    st = None if fresh else {"h": rng.standard_normal((S, N, P)), "phi": rng.uniform(-3, 3, (S, N // 2)),
                             "prev_B": rng.standard_normal((S, R, N)), "prev_x": rng.standard_normal((S, R, P))}
    ref = G.grads(x, Bm, Cm, dt, A, lam, theta, dy, dhT, st)
    for i in range(S):
        z = lambda k, shp: st[k][i] if st is not None else np.zeros(shp)
        g = backward_chunked(x[i], Bm[i], Cm[i], dt[i], A[i], lam[i], theta[i], dy[i], dhT[i],
                             z("h", (N, P)), z("phi", (N // 2,)), z("prev_B", (R, N)), z("prev_x", (R, P)), c)
        for k in ("x", "Bm", "Cm", "dt", "lam", "theta", "A", "h0"):
            assert np.max(np.abs(np.asarray(g[k]) - ref[k][i])) < 1e-9, k


def _rot_neg(cs, sn, Z):
    """R(-a) on the row pairs of a state Z [N, P]: (c u - s v, s u + c v)."""
    out = np.empty_like(Z)
    u, v = Z[0::2], Z[1::2]
    out[0::2] = cs[:, None] * u - sn[:, None] * v
    out[1::2] = sn[:, None] * u + cs[:, None] * v
    return out


def _rot_pos(cs, sn, Z):
    """R(a) on the row pairs of Z: (c u + s v, -s u + c v)."""
    return _rot_neg(cs, -sn, Z)


def backward_chunk_frames(x, Bm, Cm, dt, A, lam, theta, dy, dhT, h0, phi0, pB0, px0, c):
    """The same adjoint organised as the CUDA backward is: every chunk in its own frame (B~, C~
    rotated by the angle psi accumulated from the chunk's start), the chunk's own state terms
    dH = sum_s wx_s B~_s^T X_s and dG = sum_i exp(ell_i) C~_i^T dY_i (wx_s = Mh[last, s], plus
    q of the next chunk's first token on the last token), scans from chunk to chunk that turn
    a state by the chunk's angle advance sigma (Hp(k+1) = R(-sigma_k)(exp(ell_last) Hp(k) +
    dH(k)), Gout(k-1) = R(sigma_{k-1})(exp(ell_last) Gout(k) + dG(k))), then each chunk's
    adjoint from its Hp and Gout alone; the fold gradient of a chunk's first token comes from
    the previous chunk (<Gout, B~_last^T X_last>), d phi sums of later chunks are added last."""
    T, R, P = x.shape
    N = Bm.shape[-1]
    K = N // 2
    q = (1 - lam) * dt
    gam = lam * dt
    a = dt * A
    nch = (T + c - 1) // c
    wrap = lambda v: v - 2 * np.pi * np.round(v / (2 * np.pi))
    L = []
    for k in range(nch):
        t0, t1 = k * c, min(T, (k + 1) * c)
        n = t1 - t0
        psi = np.cumsum(dt[t0:t1, None] * theta[t0:t1], axis=0)
        cs, sn = np.cos(psi), np.sin(psi)
        Bt = rot_t(cs[:, None, :], sn[:, None, :], Bm[t0:t1])
        Ct = rot_t(cs[:, None, :], sn[:, None, :], Cm[t0:t1])
        ell = np.cumsum(a[t0:t1])
        el = np.exp(ell)
        qn = q[t1] if t1 < T else 0.0
        wx = np.array([np.exp(ell[-1] - ell[s]) * (gam[t0 + s] + q[t0 + s + 1]) if s < n - 1
                       else gam[t1 - 1] + qn for s in range(n)])
        L.append(dict(t0=t0, t1=t1, n=n, cs=cs, sn=sn, Bt=Bt, Ct=Ct, ell=ell, el=el, wx=wx,
                      dH=np.einsum("s,srn,srp->np", wx, Bt, x[t0:t1]),
                      dG=np.einsum("i,irn,irp->np", el, Ct, dy[t0:t1]),
                      sig=wrap(psi[-1]), dec=el[-1]))
    # scans between chunk frames
    c0, s0 = np.cos(phi0), np.sin(phi0)
    Hp = [None] * nch
    H = _rot_neg(c0, s0, h0) + q[0] * pB0.T @ px0
    for k in range(nch):
        Hp[k] = H
        H = _rot_neg(np.cos(L[k]["sig"]), np.sin(L[k]["sig"]), L[k]["dec"] * H + L[k]["dH"])
    ph = phi0 + sum(L[k]["sig"] for k in range(nch - 1))
    Go = [None] * nch
    G = _rot_neg(np.cos(ph), np.sin(ph), dhT)
    for k in reversed(range(nch)):
        Go[k] = G
        Y = L[k]["dec"] * G + L[k]["dG"]
        if k > 0:
            G = _rot_pos(np.cos(L[k - 1]["sig"]), np.sin(L[k - 1]["sig"]), Y)
        else:
            dHp0 = Y
    dh0 = _rot_pos(c0, s0, dHp0)
    dX = np.zeros_like(x); dB = np.zeros_like(Bm); dC = np.zeros_like(Cm)
    ddt = np.zeros(T); dlam = np.zeros(T); dtheta = np.zeros((T, K))
    dqf = np.zeros(nch)
    dqf[0] = np.sum(dHp0 * (pB0.T @ px0))
    Sphi = np.zeros((nch, K))
    dA = 0.0
    for k in range(nch):
        d = L[k]
        t0, t1, n = d["t0"], d["t1"], d["n"]
        Bt, Ct, Xc, dYc, ell, el, wx = d["Bt"], d["Ct"], x[t0:t1], dy[t0:t1], d["ell"], d["el"], d["wx"]
        ex = np.zeros((n, n)); Mh = np.zeros((n, n))
        for i in range(n):
            for s_ in range(i + 1):
                ex[i, s_] = np.exp(ell[i] - ell[s_])
                Mh[i, s_] = gam[t0 + i] if s_ == i else ex[i, s_] * (gam[t0 + s_] + q[t0 + s_ + 1])
        S = np.einsum("irn,sun->irsu", Ct, Bt)
        E = np.einsum("irp,sup->irsu", dYc, Xc)
        W = np.einsum("srn,np->srp", Bt, Go[k])
        Q = np.einsum("irp,np->irn", dYc, Hp[k])
        XG = np.einsum("srp,np->srn", Xc, Go[k])
        wdot = np.einsum("srp,srp->s", W, Xc)
        dexp = np.einsum("irn,irn->i", Ct, Q)
        dexp[n - 1] += np.sum(Go[k] * Hp[k])
        dM = np.einsum("irsu,irsu->is", S, E) * np.tri(n)
        dM[n - 1] += wdot
        MS = S * Mh[:, None, :, None]
        ME = E * Mh[:, None, :, None]
        dCt = np.einsum("irsu,sun->irn", ME, Bt) + el[:, None, None] * Q
        dBt = np.einsum("irsu,irn->sun", ME, Ct) + wx[:, None, None] * XG
        dX[t0:t1] = np.einsum("irsu,irp->sup", MS, dYc) + wx[:, None, None] * W
        dell = dexp * el
        dgam = np.zeros(n); dq = np.zeros(n)
        for t in range(n):
            dell[t] += sum(dM[t, s_] * Mh[t, s_] for s_ in range(t))
            for ti in range(t + 1, n):
                dell[t] -= dM[ti, t] * Mh[ti, t]
                dgam[t] += dM[ti, t] * ex[ti, t]
            dgam[t] += dM[t, t]
            if t > 0:
                dq[t] = sum(dM[ti, t - 1] * ex[ti, t - 1] for ti in range(t, n))
        cs, sn = d["cs"], d["sn"]
        dB[t0:t1, :, 0::2] = cs[:, None] * dBt[..., 0::2] - sn[:, None] * dBt[..., 1::2]
        dB[t0:t1, :, 1::2] = sn[:, None] * dBt[..., 0::2] + cs[:, None] * dBt[..., 1::2]
        dC[t0:t1, :, 0::2] = cs[:, None] * dCt[..., 0::2] - sn[:, None] * dCt[..., 1::2]
        dC[t0:t1, :, 1::2] = sn[:, None] * dCt[..., 0::2] + cs[:, None] * dCt[..., 1::2]
        dphi = np.sum(dBt[..., 0::2] * Bt[..., 1::2] - dBt[..., 1::2] * Bt[..., 0::2]
                      + dCt[..., 0::2] * Ct[..., 1::2] - dCt[..., 1::2] * Ct[..., 0::2], axis=1)
        g = np.cumsum(dphi[::-1], axis=0)[::-1]
        dtheta[t0:t1] = dt[t0:t1, None] * g
        Sphi[k] = g[0]
        da = np.cumsum(dell[::-1])[::-1]
        ddt[t0:t1] = np.sum(theta[t0:t1] * g, axis=1) + da * A + lam[t0:t1] * dgam + (1 - lam[t0:t1]) * dq
        dlam[t0:t1] = dt[t0:t1] * (dgam - dq)
        dA += float(np.sum(da * dt[t0:t1]))
        if k + 1 < nch:
            dqf[k + 1] = wdot[n - 1]
    for k in range(nch):
        t0, t1 = L[k]["t0"], L[k]["t1"]
        carry = Sphi[k + 1:].sum(axis=0)
        dtheta[t0:t1] += dt[t0:t1, None] * carry
        ddt[t0:t1] += theta[t0:t1] @ carry
        ddt[t0] += (1 - lam[t0]) * dqf[k]
        dlam[t0] -= dt[t0] * dqf[k]
    return dict(x=dX, Bm=dB, Cm=dC, dt=ddt, lam=dlam, theta=dtheta, A=dA, h0=dh0)


@pytest.mark.parametrize("T,N,P,R,c,fresh", [(7, 4, 3, 1, 3, True), (11, 6, 5, 2, 4, False),
                                            (9, 4, 2, 4, 2, False), (12, 8, 4, 1, 12, False),
                                            (5, 4, 3, 2, 1, False), (23, 8, 6, 1, 4, False)])
def test_chunk_frames_decomposition_equals_gradient_oracle(T, N, P, R, c, fresh):
    rng = np.random.Generator(np.random.PCG64(T * 100 + N * 10 + R + 7))
    S = 2
    x = rng.standard_normal((S, T, R, P))
    Bm = rng.standard_normal((S, T, R, N)) / np.sqrt(N)
    Cm = rng.standard_normal((S, T, R, N)) / np.sqrt(N)
    dt = rng.uniform(0.05, 0.6, (S, T))
    A = -rng.uniform(0.5, 3, S)
    lam = rng.uniform(0, 1, (S, T))
    theta = rng.standard_normal((S, T, N // 2)) * 3
    dy = rng.standard_normal((S, T, R, P))
    dhT = rng.standard_normal((S, N, P))
    st = None if fresh else {"h": rng.standard_normal((S, N, P)), "phi": rng.uniform(-3, 3, (S, N // 2)),
                             "prev_B": rng.standard_normal((S, R, N)), "prev_x": rng.standard_normal((S, R, P))}
    ref = G.grads(x, Bm, Cm, dt, A, lam, theta, dy, dhT, st)
    for i in range(S):
        z = lambda k, shp: st[k][i] if st is not None else np.zeros(shp)
        g = backward_chunk_frames(x[i], Bm[i], Cm[i], dt[i], A[i], lam[i], theta[i], dy[i], dhT[i],
                                  z("h", (N, P)), z("phi", (N // 2,)), z("prev_B", (R, N)),
                                  z("prev_x", (R, P)), c)
        for k in ("x", "Bm", "Cm", "dt", "lam", "theta", "A", "h0"):
            assert np.max(np.abs(np.asarray(g[k]) - ref[k][i])) < 1e-9, k
