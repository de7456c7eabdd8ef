"""fp64 numpy model of the chunked forms the CUDA kernels implement.

This is not the oracle: it is the blocked algebra the kernels follow, written
plainly so that a test can hold it against the sequential oracle in fp64.  It
shares no code with either.

Q-Delta (reading notes "Q-Delta: Beyond Key-Value Associative State Evolution",
sec. 3.3.2, Eqs. 20-27, with the notes' corrections of the v1 transposes and the
missing gamma_r/gamma_i decay).  Per chunk of C tokens, with rows stacked,
l_i = sum_{j<=i} log alpha_j, gamma_i = exp(l_i), X = K + diag(lambda) Q,
H_ij = exp(l_i - l_j) for j <= i:
    A     = strictly_lower(diag(beta) (H * X K^T))
    Z     = (I + A)^{-1} (diag(beta) V - diag(beta gamma) X S_in^T)
    O     = diag(gamma) Q S_in^T + (H * Q K^T) Z            (H includes the diagonal)
    S_out = gamma_C S_in + Z^T diag(exp(l_C - l_i)) K
The single solve is the notes' pair of UT solves folded together
((I + L_gamma)^{-1} = D_gamma (I + L)^{-1} D_gamma^{-1}).

QED (reading notes "The Query Knows What to Forget", sec. 2.2, Eq. 6 and the
GDN-2 update of Eqs. 4/8), with the state stored as its transpose S^ (V x K),
per-channel cumulative log-decay G_i = sum_{j<=i} g_j (vectors over K),
a_i = b_i*k_i + lambda_h (u_i - k_i (k_i^T u_i)), u_i = b_i*q_i:
    At    = strictly_lower((A*e^G)(K*e^-G)^T)
    Z     = (I + At)^{-1} (W*V - (A*e^G) S^_in^T)
    O     = (Q*e^G) S^_in^T + incl_lower((Q*e^G)(K*e^-G)^T) Z
    S^out = S^_in diag(e^{G_C}) + Z^T (K*e^{G_C - G})
"""
import numpy as np


def qdelta_chunked(q, k, v, alpha, beta, lam, S0, C=64):
    """One stream: q, k [T,dk]; v [T,dv]; gates [T] (None: alpha=1 / lam=0);
    S0 [dv,dk] or None.  Returns (o [T,dv], S_final [dv,dk])."""
    T, dk = q.shape
    dv = v.shape[1]
    S = np.zeros((dv, dk)) if S0 is None else np.array(S0, dtype=np.float64)
    alpha = np.ones(T) if alpha is None else alpha
    lam = np.zeros(T) if lam is None else lam
    o = np.zeros((T, dv))
    for c0 in range(0, T, C):
        c1 = min(T, c0 + C)
        n = c1 - c0
        Q, K, V = q[c0:c1], k[c0:c1], v[c0:c1]
        bt, lm = beta[c0:c1], lam[c0:c1]
        ell = np.cumsum(np.log(alpha[c0:c1]))
        X = K + lm[:, None] * Q
        Hm = np.tril(np.exp(ell[:, None] - ell[None, :]))
        A = np.tril(bt[:, None] * Hm * (X @ K.T), -1)
        Z = np.linalg.solve(np.eye(n) + A, bt[:, None] * V - (bt * np.exp(ell))[:, None] * (X @ S.T))
        o[c0:c1] = np.exp(ell)[:, None] * (Q @ S.T) + (Hm * (Q @ K.T)) @ Z
        S = np.exp(ell[-1]) * S + Z.T @ (np.exp(ell[-1] - ell)[:, None] * K)
    return o, S


def qed_chunked(q, k, v, g, b, w, lam_h, S0, C=64):
    """One stream: q, k, g, b [T,K]; v, w [T,V]; lam_h scalar; S0 [V,K] (S^) or None."""
    T, K = q.shape
    V = v.shape[1]
    S = np.zeros((V, K)) if S0 is None else np.array(S0, dtype=np.float64)
    o = np.zeros((T, V))
    for c0 in range(0, T, C):
        c1 = min(T, c0 + C)
        n = c1 - c0
        Qc, Kc, Vc, bc, wc = q[c0:c1], k[c0:c1], v[c0:c1], b[c0:c1], w[c0:c1]
        G = np.cumsum(g[c0:c1], axis=0)
        u = bc * Qc
        d = u - Kc * np.sum(Kc * u, axis=1, keepdims=True)
        A = bc * Kc + lam_h * d
        Ae, Qe, Ke = A * np.exp(G), Qc * np.exp(G), Kc * np.exp(-G)
        At = np.tril(Ae @ Ke.T, -1)
        Z = np.linalg.solve(np.eye(n) + At, wc * Vc - Ae @ S.T)
        o[c0:c1] = Qe @ S.T + np.tril(Qe @ Ke.T) @ Z
        S = S * np.exp(G[-1])[None, :] + Z.T @ (Kc * np.exp(G[-1][None, :] - G))
    return o, S


def qdelta_chunked_bwd(q, k, v, alpha, beta, lam, S0, dO, dS_final, C=64):
    """Backward of qdelta_chunked for one stream, chunk by chunk in reverse, the
    algebra the CUDA backward implements.  Chunk-entry states come from a forward
    sweep.  Per chunk, with the forward's names plus XS = diag(gamma) X S_in^T,
    QS = diag(gamma) Q S_in^T, P = H * Q K^T, M = strictly_lower(H * X K^T),
    w_i = exp(l_C - l_i), T = (I + diag(beta) M)^{-1}, Z = T diag(beta) (V - XS):
        dZ  = P^T dO + diag(w) K dS_out^T           dR = T^T dZ
        dA  = -strictly_lower(dR Z^T)               dM = diag(beta) dA
        dP  = lower(dO Z^T)                          dXS = -diag(beta) dR
        dV  = diag(beta) dR
        dbeta = rowsum(dA * M) + rowsum(dR * (V - XS))
        dS_in = gamma_C dS_out + (gamma * dO)^T Q + (gamma * dXS)^T X
        dQ  = (gamma * dO) S_in + (H * dP) K + lambda dX
        dX  = (gamma * dXS) S_in + (H * dM) K
        dK  = (H * dP)^T Q + (H * dM)^T X + diag(w) Z dS_out + dX
        dlambda = rowsum(dX * Q)
        dl  = rowsum(dO * QS) + rowsum(dXS * XS) + rowsum(E) - colsum(E) - wz
              (+ gamma_C <dS_out, S_in> + sum(wz) on the chunk's last token)
        with E = dP * P + dM * M and wz_i = w_i (Z dS_out)_i . K_i;
        d log alpha = reverse cumsum of dl over the chunk; dalpha = d log alpha / alpha.
    Returns dq, dk, dv, dalpha (None if alpha is None), dbeta, dlam (None if lam is
    None), dS0."""
    T, dk = q.shape
    dv = v.shape[1]
    al = np.ones(T) if alpha is None else alpha
    lm = np.zeros(T) if lam is None else lam
    S = np.zeros((dv, dk)) if S0 is None else np.array(S0, dtype=np.float64)
    starts = list(range(0, T, C))
    S_in = []
    for c0 in starts:                                     # forward sweep: chunk-entry states
        S_in.append(S.copy())
        c1 = min(T, c0 + C)
        _, S = qdelta_chunked(q[c0:c1], k[c0:c1], v[c0:c1], al[c0:c1], beta[c0:c1], lm[c0:c1], S, C)
    dq, dkk, dvv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    dlog, dbeta, dlam = np.zeros(T), np.zeros(T), np.zeros(T)
    dS = np.zeros((dv, dk)) if dS_final is None else np.array(dS_final, dtype=np.float64)
    for ci in range(len(starts) - 1, -1, -1):
        c0 = starts[ci]
        c1 = min(T, c0 + C)
        n = c1 - c0
        Si = S_in[ci]
        Q, K, V, b, lc, dOc = q[c0:c1], k[c0:c1], v[c0:c1], beta[c0:c1], lm[c0:c1], dO[c0:c1]
        ell = np.cumsum(np.log(al[c0:c1]))
        gam, gC = np.exp(ell), np.exp(ell[-1])
        w = np.exp(ell[-1] - ell)
        X = K + lc[:, None] * Q
        Hm = np.tril(np.exp(ell[:, None] - ell[None, :]))
        P = Hm * (Q @ K.T)
        M = np.tril(Hm * (X @ K.T), -1)
        Tm = np.linalg.inv(np.eye(n) + b[:, None] * M)
        XS, QS = gam[:, None] * (X @ Si.T), gam[:, None] * (Q @ Si.T)
        Z = Tm @ (b[:, None] * (V - XS))
        dZ = P.T @ dOc + (w[:, None] * K) @ dS.T
        dR = Tm.T @ dZ
        dA = -np.tril(dR @ Z.T, -1)
        dM = b[:, None] * dA
        dP = np.tril(dOc @ Z.T)
        dXS = -b[:, None] * dR
        dvv[c0:c1] = b[:, None] * dR
        dbeta[c0:c1] = (dA * M).sum(1) + (dR * (V - XS)).sum(1)
        dX = (gam[:, None] * dXS) @ Si + (Hm * dM) @ K
        dq[c0:c1] = (gam[:, None] * dOc) @ Si + (Hm * dP) @ K + lc[:, None] * dX
        ZdS = Z @ dS
        dkk[c0:c1] = (Hm * dP).T @ Q + (Hm * dM).T @ X + w[:, None] * ZdS + dX
        dlam[c0:c1] = (dX * Q).sum(1)
        E = dP * P + dM * M
        wz = w * (ZdS * K).sum(1)
        dl = (dOc * QS).sum(1) + (dXS * XS).sum(1) + E.sum(1) - E.sum(0) - wz
        dl[-1] += gC * (dS * Si).sum() + wz.sum()
        dlog[c0:c1] = np.cumsum(dl[::-1])[::-1]
        dS = gC * dS + (gam[:, None] * dOc).T @ Q + (gam[:, None] * dXS).T @ X
    return {"dq": dq, "dk": dkk, "dv": dvv, "dalpha": None if alpha is None else dlog / alpha,
            "dbeta": dbeta, "dlam": None if lam is None else dlam, "dS0": dS}
