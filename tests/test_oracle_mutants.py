"""The pins are discriminative: plausible mistakes in a recurrence fail them.

Each mutant is a one-step recurrence with one planted mistake (CPU only, never
the GPU path).  The same pin predicates that the oracle passes must reject every
mutant, so a mistake of that kind in the oracle could not go unnoticed.
"""
import json
import os

import numpy as np
import pytest

import oracle

rng = np.random.default_rng(99)


def _unit(x):
    return x / np.linalg.norm(x)


def oracle_qdelta_step(Sp, q, k, v, al, be, lm):
    sh = lambda x: np.asarray(x, dtype=np.float64).reshape(1, 1, 1, -1)
    g = lambda x: np.array([[[x]]])
    o, S = oracle.qdelta_fwd(sh(q), sh(k), sh(v), g(al), g(be), g(lm), Sp[None, None])
    return S[0, 0], o[0, 0, 0]


def _qdelta_mutant(kind):
    def step(Sp, q, k, v, al, be, lm):
        x = k + lm * q
        Sb = al * Sp
        if kind == "normalised_residual":
            e = (v - Sb @ x) / (1 + lm)
        elif kind == "decay_after_error":
            e = v - Sp @ x
        elif kind == "lambda_sign":
            e = v - Sb @ (k - lm * q)
        else:
            e = v - Sb @ x
        w = x if kind == "write_along_x" else k
        S = Sb + be * np.outer(e, w)
        o = Sb @ q if kind == "output_before_update" else S @ q
        return S, o
    return step


def qdelta_pins_hold(step):
    """Gated error identity and closed-form output (Q-Delta notes sec. 2.4, 2.7)."""
    dk, dv = 6, 5
    for _ in range(5):
        q, k = _unit(rng.standard_normal(dk)), _unit(rng.standard_normal(dk))
        v = rng.standard_normal(dv)
        al, be, lm = rng.uniform(0.8, 0.99), rng.uniform(0.1, 0.9), rng.uniform(0.1, 0.9)
        Sp = rng.standard_normal((dv, dk))
        S, o = step(Sp, q, k, v, al, be, lm)
        x = k + lm * q
        ok1 = np.allclose(v - S @ x, (1 - be * (k @ x)) * (v - al * Sp @ x), atol=1e-10)
        ok2 = np.allclose(o, al * Sp @ q + be * (v - al * Sp @ x) * (k @ q), atol=1e-10)
        if not (ok1 and ok2):
            return False
    return True


def test_oracle_passes_qdelta_pins():
    assert qdelta_pins_hold(oracle_qdelta_step)


@pytest.mark.parametrize("kind", ["normalised_residual", "decay_after_error", "lambda_sign",
                                  "write_along_x", "output_before_update"])
def test_qdelta_mutant_rejected(kind):
    assert not qdelta_pins_hold(_qdelta_mutant(kind))


def oracle_qed_step(Sbar, q, k, b, w, v, lam):
    K, V = Sbar.shape
    sh = lambda x: np.asarray(x, dtype=np.float64).reshape(1, 1, 1, -1)
    o, S = oracle.qed_fwd(sh(q), sh(k), sh(v), sh(np.zeros(K)), sh(b), sh(w), np.array([lam]),
                          Sbar.T.reshape(1, 1, V, K))
    return S[0, 0].T, o[0, 0, 0]


def _qed_mutant(kind):
    def step(Sbar, q, k, b, w, v, lam):
        if kind == "no_projection":
            d = b * q
        elif kind == "project_then_gate":
            d = b * (q - k * (k @ q))
        elif kind == "ungated_query":
            d = q - k * (k @ q)
        else:
            u = b * q
            d = u - k * (k @ u)
        a = b * k + lam * d
        if kind == "lambda_on_base":
            a = lam * b * k + d
        r = w * v - Sbar.T @ a
        S = Sbar + np.outer(k, r)
        return S, S.T @ q
    return step


def qed_pins_hold(step):
    """Printed 2-D example and Eqs. 11-12 (QED notes sec. 2.3-2.4)."""
    ex = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "qed_2d_example.json")))
    i, e = ex["inputs"], ex["expected"]
    S, o = step(np.array(i["S_bar_KxV"]), np.array(i["q"]), np.array(i["k"]), np.array(i["b"]),
                np.ones(1), np.array([i["w_times_v"]]), i["lambda_h"])
    if abs(o - e["o_qed"]) > 1e-12:
        return False
    K, V = 6, 4
    for _ in range(3):
        q, k = _unit(rng.standard_normal(K)), _unit(rng.standard_normal(K))
        b, w = rng.uniform(0.1, 0.9, K), rng.uniform(0.1, 0.9, V)
        v, Sbar, lam = rng.standard_normal(V), rng.standard_normal((K, V)), 0.45
        Sq, oq = step(Sbar, q, k, b, w, v, lam)
        Sg, og = step(Sbar, q, k, b, w, v, 0.0)
        u = b * q
        d = u - k * (k @ u)
        if not np.allclose(Sq - Sg, -lam * np.outer(k, Sbar.T @ d), atol=1e-10):
            return False
        if not np.allclose(oq - og, -lam * (q @ k) * (Sbar.T @ d), atol=1e-10):
            return False
    return True


def test_oracle_passes_qed_pins():
    assert qed_pins_hold(oracle_qed_step)


@pytest.mark.parametrize("kind", ["no_projection", "project_then_gate", "ungated_query",
                                  "lambda_on_base"])
def test_qed_mutant_rejected(kind):
    assert not qed_pins_hold(_qed_mutant(kind))


# the QED ablation arms (QED notes, sec. 3.2, Table 1): new erase term t added to b*k
_ARM_2D = {"nogate": (1.52, 3.312), "nogate_noproj": (1.28, 3.168), "rand": (1.70, 3.42)}


def oracle_qed_arm_step(arm):
    def step(Sbar, q, k, b, w, v, lam, z):
        K, V = Sbar.shape
        sh = lambda x: np.asarray(x, dtype=np.float64).reshape(1, 1, 1, -1)
        o, S = oracle.qed_fwd_variant(sh(q), sh(k), sh(v), sh(np.zeros(K)), sh(b), sh(w), np.array([lam]), arm,
                                      np.asarray(z, dtype=np.float64).reshape(1, K), Sbar.T.reshape(1, 1, V, K))
        return S[0, 0].T, o[0, 0, 0]
    return step


def _qed_arm_mutant(arm, kind):
    def step(Sbar, q, k, b, w, v, lam, z):
        P = lambda u: u - k * (k @ u)
        t = {"nogate": P(q), "nogate_noproj": q, "rand": P(b * z)}[arm]
        if kind == "gate_kept":
            t = P(b * q) if arm != "rand" else P(b * q)
        elif kind == "projection_kept":
            t = P(q) if arm == "nogate_noproj" else t
        elif kind == "rand_ungated":
            t = P(z) if arm == "rand" else t
        a = b * k + lam * t
        r = w * v - Sbar.T @ a
        S = Sbar + np.outer(k, r)
        return S, S.T @ q
    return step


def qed_arm_pins_hold(arm, step):
    """The arm's hand-derived values on the sec. 2.4 example, and Eqs. 11-12 with
    the arm's own new term."""
    S1, o1 = _ARM_2D[arm]
    S, o = step(np.array([[2.0], [3.0]]), np.array([0.6, 0.8]), np.array([1.0, 0.0]), np.array([0.5, 0.5]),
                np.ones(1), np.ones(1), 0.2, np.array([0.0, 1.0]))
    if abs(o - o1) > 1e-12 or abs(S[0, 0] - S1) > 1e-12:
        return False
    K, V = 6, 4
    for _ in range(3):
        q, k, z = _unit(rng.standard_normal(K)), _unit(rng.standard_normal(K)), _unit(rng.standard_normal(K))
        b, w = rng.uniform(0.1, 0.9, K), rng.uniform(0.1, 0.9, V)
        v, Sbar, lam = rng.standard_normal(V), rng.standard_normal((K, V)), 0.45
        Sa, oa = step(Sbar, q, k, b, w, v, lam, z)
        Sg, og = step(Sbar, q, k, b, w, v, 0.0, z)
        P = lambda u: u - k * (k @ u)
        t = {"nogate": P(q), "nogate_noproj": q, "rand": P(b * z)}[arm]
        if not np.allclose(Sa - Sg, -lam * np.outer(k, Sbar.T @ t), atol=1e-10):
            return False
    return True


@pytest.mark.parametrize("arm", ["nogate", "nogate_noproj", "rand"])
def test_oracle_passes_qed_arm_pins(arm):
    assert qed_arm_pins_hold(arm, oracle_qed_arm_step(arm))


@pytest.mark.parametrize("arm,kind", [("nogate", "gate_kept"), ("nogate_noproj", "projection_kept"),
                                      ("nogate_noproj", "gate_kept"), ("rand", "gate_kept"),
                                      ("rand", "rand_ungated")])
def test_qed_arm_mutant_rejected(arm, kind):
    assert not qed_arm_pins_hold(arm, _qed_arm_mutant(arm, kind))


# the prologue (DeltaNet notes sec. 3.8; Q-Delta notes sec. 2.5): feature map and gates
def _prologue_mutant(kind):
    def fmap(x):
        s = x * (1.0 / (1.0 + np.exp(x))) if kind == "silu_sign" else x / (1.0 + np.exp(-x))
        n = np.abs(s).sum(-1, keepdims=True) if kind == "l1_norm" else np.linalg.norm(s, axis=-1, keepdims=True)
        return s / n
    def gate_alpha(x):
        return 1.0 / (1.0 + np.exp(-x)) if kind == "alpha_sigmoid" else np.exp(-np.log1p(np.exp(x)))
    def fwd(q_raw, k_raw, v, a_l, b_l, l_l, S0):
        return oracle.qdelta_fwd(fmap(q_raw), fmap(k_raw), v, gate_alpha(a_l), 1.0 / (1.0 + np.exp(-b_l)),
                                 1.0 / (1.0 + np.exp(-l_l)), S0)
    return fwd


def oracle_prologue(q_raw, k_raw, v, a_l, b_l, l_l, S0):
    return oracle.qdelta_fwd_prologue(q_raw, k_raw, v, a_l, b_l, l_l, S0)


def prologue_pins_hold(fwd):
    """SiLU's shape on (ln 3, -ln 3) -> (3, -1)/sqrt(10) and alpha = 1/(1 + e^x)."""
    T, H = 3, 2
    l3 = np.log(3.0)
    raw = np.broadcast_to(np.array([l3, -l3, 0.0, 0.0]), (1, T, H, 4)).copy()
    feat = np.broadcast_to(np.array([3.0, -1.0, 0.0, 0.0]) / np.sqrt(10.0), (1, T, H, 4)).copy()
    v = rng.standard_normal((1, T, H, 4))
    a_l = rng.uniform(-3, 3, (1, T, H))
    b_l = rng.uniform(-3, 3, (1, T, H))
    l_l = rng.uniform(-3, 3, (1, T, H))
    S0 = rng.standard_normal((1, H, 4, 4)) * 0.3
    o1, S1 = fwd(raw, raw, v, a_l, b_l, l_l, S0)
    o2, S2 = oracle.qdelta_fwd(feat, feat, v, 1.0 / (1.0 + np.exp(a_l)), 1.0 / (1.0 + np.exp(-b_l)),
                               1.0 / (1.0 + np.exp(-l_l)), S0)
    return np.allclose(o1, o2, atol=1e-12) and np.allclose(S1, S2, atol=1e-12)


def test_oracle_passes_prologue_pins():
    assert prologue_pins_hold(oracle_prologue)


@pytest.mark.parametrize("kind", ["silu_sign", "l1_norm", "alpha_sigmoid"])
def test_prologue_mutant_rejected(kind):
    assert not prologue_pins_hold(_prologue_mutant(kind))


# ---------------------------------------------------------------- backward

def _bwd_rowwise(kind=None):
    """Single-stream adjoint (B = H = 1), row by row, with an optional planted mistake."""
    def bwd(q, k, v, al, be, lm, S0, dO, dS):
        T, dk = q.shape
        dv = v.shape[1]
        x = k + lm[:, None] * q
        g = {"dq": np.zeros_like(q), "dk": np.zeros_like(k), "dv": np.zeros_like(v),
             "dalpha": np.zeros(T), "dbeta": np.zeros(T), "dlam": np.zeros(T), "dS0": np.zeros_like(S0)}
        for i in range(dv):
            hist, e = [S0[i].copy()], np.zeros(T)
            for t in range(T):
                sb = al[t] * hist[-1]
                e[t] = v[t, i] - sb @ x[t]
                hist.append(sb + be[t] * e[t] * k[t])
            gs = dS[i].copy()
            for t in range(T - 1, -1, -1):
                gs = gs + dO[t, i] * q[t]
                g["dq"][t] += dO[t, i] * hist[t + 1]
                gk = gs @ k[t]
                ge = be[t] * gk
                g["dbeta"][t] += (v[t, i] if kind == "dbeta_uses_value" else e[t]) * gk
                if kind != "dk_drops_write_term":
                    g["dk"][t] += be[t] * e[t] * gs
                g["dv"][t, i] = ge
                gbar = gs - ge * x[t]
                dx = (1 if kind == "dx_sign" else -1) * ge * al[t] * hist[t]
                g["dk"][t] += dx
                if kind != "dq_drops_lambda_term":
                    g["dq"][t] += lm[t] * dx
                g["dlam"][t] += q[t] @ dx
                g["dalpha"][t] += gbar @ (hist[t + 1] if kind == "dalpha_new_state" else hist[t])
                gs = gbar if kind == "carry_without_decay" else al[t] * gbar
            g["dS0"][i] = gs
        return g
    return bwd


def backward_pins_hold(bwd):
    """Central differences of the pinned forward oracle (the backward's pin)."""
    T, dk, dv = 6, 4, 3
    q, k = rng.standard_normal((T, dk)), rng.standard_normal((T, dk))
    v = rng.standard_normal((T, dv))
    al, be, lm = rng.uniform(0.5, 1.0, T), rng.uniform(0.1, 0.9, T), rng.uniform(0.1, 0.9, T)
    S0, dS = rng.standard_normal((dv, dk)), rng.standard_normal((dv, dk))
    dO = rng.standard_normal((T, dv))
    g = bwd(q, k, v, al, be, lm, S0, dO, dS)
    ex = lambda a: a[None, :, None]
    args = {"q": q, "k": k, "v": v, "alpha": al, "beta": be, "lam": lm, "S0": S0}

    def loss(a):
        o, S = oracle.qdelta_fwd(ex(a["q"]), ex(a["k"]), ex(a["v"]), ex(a["alpha"]), ex(a["beta"]),
                                 ex(a["lam"]), a["S0"][None, None])
        return (o[0, :, 0] * dO).sum() + (S[0, 0] * dS).sum()

    for name, x in args.items():
        for idx in np.ndindex(x.shape):
            a = dict(args)
            xp, xm = x.copy(), x.copy()
            xp[idx] += 1e-6
            xm[idx] -= 1e-6
            a[name] = xp
            lp = loss(a)
            a[name] = xm
            fd = (lp - loss(a)) / 2e-6
            if abs(g["d" + name][idx] - fd) > 1e-6 * max(1.0, abs(fd)):
                return False
    return True


def test_oracle_and_rowwise_adjoint_pass_backward_pins():
    def via_oracle(q, k, v, al, be, lm, S0, dO, dS):
        ex = lambda a: a[None, :, None]
        g = oracle.qdelta_bwd(ex(q), ex(k), ex(v), ex(al), ex(be), ex(lm), S0[None, None], ex(dO), dS[None, None])
        return {n: (a[0, :, 0] if n != "dS0" else a[0, 0]) for n, a in g.items()}
    assert backward_pins_hold(via_oracle)
    assert backward_pins_hold(_bwd_rowwise())


@pytest.mark.parametrize("kind", ["dbeta_uses_value", "dk_drops_write_term", "dx_sign", "dq_drops_lambda_term",
                                  "dalpha_new_state", "carry_without_decay"])
def test_backward_mutant_rejected(kind):
    assert not backward_pins_hold(_bwd_rowwise(kind))


# ---------------------------------------------------------------- EDA

def oracle_eda_step(Sp, q, k, v, e, be):
    sh = lambda x: np.asarray(x, dtype=np.float64).reshape(1, 1, 1, -1)
    o, S = oracle.eda_fwd(sh(q), sh(k), sh(v), sh(e), np.array([[[be]]]), Sp[None, None])
    return S[0, 0], o[0, 0, 0]


def _eda_mutant(kind):
    def step(Sp, q, k, v, e, be):
        P = np.eye(len(e)) - (2.0 if kind == "reflection" else 1.0) * np.outer(e, e)
        Se = Sp @ P
        if kind == "erase_after_write":
            S = (Sp - be * np.outer(Sp @ k - v, k)) @ P
        elif kind == "residual_before_erase":
            S = Se - be * np.outer(Sp @ k - v, k)
        elif kind == "erase_along_key":
            S = (Sp @ (np.eye(len(e)) - np.outer(k, k))) - be * np.outer(Sp @ k - v, k)
        else:
            S = Se - be * np.outer(Se @ k - v, k)
        o = Se @ q if kind == "output_before_write" else S @ q
        return S, o
    return step


def eda_pins_hold(step):
    """Erase-only projection, unit-step retrieval, the e = k reduction to DeltaNet and
    the transition-product form A = (I - e e^T)(I - beta k k^T)."""
    d, dv = 6, 4
    for _ in range(4):
        q, k, e = (_unit(rng.standard_normal(d)) for _ in range(3))
        v = rng.standard_normal(dv)
        Sp = rng.standard_normal((dv, d))
        be = rng.uniform(0.2, 0.9)
        S, o = step(Sp, q, np.zeros(d), np.zeros(dv), e, be)
        if not np.allclose(S, Sp @ (np.eye(d) - np.outer(e, e)), atol=1e-12):
            return False
        S, o = step(Sp, q, k, v, e, 1.0)
        if not np.allclose(S @ k, v, atol=1e-12):
            return False
        S, o = step(Sp, q, k, v, k, 1.0)
        if not np.allclose(S, Sp - np.outer(Sp @ k - v, k), atol=1e-12):
            return False
        S, o = step(Sp, q, k, v, e, be)
        A = (np.eye(d) - np.outer(e, e)) @ (np.eye(d) - be * np.outer(k, k))
        if not (np.allclose(S, Sp @ A + be * np.outer(v, k), atol=1e-12) and np.allclose(o, S @ q, atol=1e-12)):
            return False
    return True


def test_oracle_passes_eda_pins():
    assert eda_pins_hold(oracle_eda_step)


@pytest.mark.parametrize("kind", ["reflection", "erase_after_write", "residual_before_erase", "erase_along_key",
                                  "output_before_write"])
def test_eda_mutant_rejected(kind):
    assert not eda_pins_hold(_eda_mutant(kind))


# ---------------------------------------------------------------- prologue backward

def _feature_map_bwd(kind=None):
    """dx of y = SiLU(x)/|SiLU(x)| for an incoming dy, with an optional planted mistake."""
    def bwd(x, dy):
        sg = 1.0 / (1.0 + np.exp(-x))
        s = x * sg
        n = np.linalg.norm(s)
        y = s / n
        ds = dy / n if kind == "no_projection" else (dy - y * (y @ dy)) / (1.0 if kind == "no_norm" else n)
        dsilu = sg if kind == "silu_derivative_is_sigmoid" else sg * (1.0 + x * (1.0 - sg))
        return ds * dsilu
    return bwd


def feature_map_bwd_pins_hold(bwd):
    """Central differences of the oracle's prologue forward at one token (T = 1, S0 = 0):
    with beta = 1, v = e_1 and dO = e_1, o = (k . q) e_1, so dL/dq_raw = J_q^T k."""
    d = 5
    for _ in range(3):
        xq, xk = rng.standard_normal(d), rng.standard_normal(d)
        sh = lambda a: np.asarray(a, dtype=np.float64).reshape(1, 1, 1, -1)
        v = np.zeros(d)
        v[0] = 1.0
        blog = np.array([[[50.0]]])                          # beta = 1 to double precision
        fwd = lambda x: oracle.qdelta_fwd_prologue(sh(x), sh(xk), sh(v), None, blog, None, None)[0][0, 0, 0, 0]
        fd = np.array([(fwd(xq + 1e-6 * np.eye(d)[i]) - fwd(xq - 1e-6 * np.eye(d)[i])) / 2e-6 for i in range(d)])
        sk = xk / (1.0 + np.exp(-xk))
        if not np.allclose(bwd(xq, sk / np.linalg.norm(sk)), fd, atol=1e-7):
            return False
    return True


def test_correct_feature_map_backward_passes_pin():
    assert feature_map_bwd_pins_hold(_feature_map_bwd())


@pytest.mark.parametrize("kind", ["no_projection", "no_norm", "silu_derivative_is_sigmoid"])
def test_feature_map_backward_mutant_rejected(kind):
    assert not feature_map_bwd_pins_hold(_feature_map_bwd(kind))
