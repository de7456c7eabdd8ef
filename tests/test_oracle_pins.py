"""Pins of the fp64 oracle to what the pages and the mathematics fix.

None of these re-types the oracle's own update: each checks it against a
printed worked example, a closed form or identity derived on the pages, a
special case that reduces to another page's formulation, an invariant, or a
brute-force expansion by explicit transition-matrix products.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(12345)


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _rand_qdelta(B, T, H, dk, dv, gated=True, lam=True, s0=True, unit=True):
    q = rng.standard_normal((B, T, H, dk))
    k = rng.standard_normal((B, T, H, dk))
    if unit:
        q, k = _unit(q), _unit(k)
    v = rng.standard_normal((B, T, H, dv))
    beta = rng.uniform(0.05, 1.0, (B, T, H))
    alpha = rng.uniform(0.8, 1.0, (B, T, H)) if gated else None
    lm = rng.uniform(0.0, 1.0, (B, T, H)) if lam else None
    S0 = rng.standard_normal((B, H, dv, dk)) * 0.3 if s0 else None
    return q, k, v, alpha, beta, lm, S0


def _states_per_step(q, k, v, alpha, beta, lam, S0):
    """S_0..S_T for a single stream (B=H=1) by carrying the oracle's state."""
    T = q.shape[1]
    dk, dv = q.shape[-1], v.shape[-1]
    S = np.zeros((1, 1, dv, dk)) if S0 is None else S0.copy()
    states, outs = [S[0, 0].copy()], []
    for t in range(T):
        sl = slice(t, t + 1)
        o, S = oracle.qdelta_fwd(q[:, sl], k[:, sl], v[:, sl],
                                 None if alpha is None else alpha[:, sl], beta[:, sl],
                                 None if lam is None else lam[:, sl], S)
        states.append(S[0, 0].copy())
        outs.append(o[0, 0, 0])
    return states, outs


# ---------------------------------------------------------------- QED (page 3)

def _qed_one_step(k, q, b, Sbar_KxV, w, v, lam_h, g=None):
    """One oracle QED step with S0 = Sbar (g = 0 unless given). Returns (S_KxV, o)."""
    K, V = Sbar_KxV.shape
    sh = lambda x: np.asarray(x, dtype=np.float64).reshape(1, 1, 1, -1)
    g = np.zeros(K) if g is None else g
    S0 = Sbar_KxV.T.reshape(1, 1, V, K)
    o, S = oracle.qed_fwd(sh(q), sh(k), sh(v), sh(g), sh(b), sh(w), np.array([lam_h]), S0)
    return S[0, 0].T, o[0, 0, 0]


def test_qed_worked_example_2d():
    """QED notes, sec. 2.4: the printed 2-D example, exactly."""
    ex = json.load(open(os.path.join(GOLDEN, "qed_2d_example.json")))
    i, e = ex["inputs"], ex["expected"]
    Sbar = np.array(i["S_bar_KxV"])
    S, o = _qed_one_step(i["k"], i["q"], i["b"], Sbar, [1.0], [i["w_times_v"]], i["lambda_h"])
    np.testing.assert_allclose(S, np.array(e["S_qed_KxV"]), rtol=0, atol=1e-14)
    assert abs(o - e["o_qed"]) < 1e-14
    np.testing.assert_allclose(S - Sbar, np.array(e["delta_S_KxV"]), atol=1e-14)
    S2, o2 = _qed_one_step(i["k"], i["q"], i["b"], Sbar, [1.0], [i["w_times_v"]], 0.0)
    assert abs(o2 - e["o_gdn2"]) < 1e-14
    np.testing.assert_allclose(S2, Sbar, atol=1e-14)   # baseline residual is exactly zero
    assert abs((o2 - o) - e["o_difference"]) < 1e-14
    # the printed decomposition 0.144 = lambda * rho * (Sbar^T d)
    rho = float(np.dot(i["q"], i["k"]))
    assert abs(i["lambda_h"] * rho * e["S_bar_T_d"] - e["o_difference"]) < 1e-14


def _erase_factor(k, q, b, lam_h, g=None):
    """M = I - k a^T read off the oracle: v = 0 and S0 = I (V = K) give S_1 = M Sbar."""
    K = len(k)
    S, _ = _qed_one_step(k, q, b, np.eye(K), np.ones(K), np.zeros(K), lam_h, g)
    return S


def test_qed_erase_factor_counterexample():
    """QED notes, sec. 2.5: M = [[0.5,-0.1],[0,1]], spec {0.5, 1}, |M e2|^2 = 1.01."""
    ex = json.load(open(os.path.join(GOLDEN, "qed_erase_factor.json")))
    i, e = ex["inputs"], ex["expected"]
    M = _erase_factor(i["k"], i["q"], i["b"], i["lambda_h"])
    np.testing.assert_allclose(M, np.array(e["M"]), atol=1e-15)
    np.testing.assert_allclose(np.sort(np.linalg.eigvals(M).real), e["spectrum"], atol=1e-14)
    assert abs(np.sum((M @ np.array([0.0, 1.0])) ** 2) - e["norm_M_e2_squared"]) < 1e-14


@pytest.mark.parametrize("lam_h", [0.0, 0.3, 1.0, 2.5])
def test_qed_erase_spectrum_independent_of_lambda(lam_h):
    """QED notes, sec. 2.5: M has K-1 unit eigenvalues and 1 - sum_i b_i k_i^2,
    whatever lambda_h (d is orthogonal to k)."""
    K = 8
    k = _unit(rng.standard_normal(K))
    q = _unit(rng.standard_normal(K))
    b = rng.uniform(0.05, 0.95, K)
    M = _erase_factor(k, q, b, lam_h)
    ev = np.sort(np.linalg.eigvals(M).real)
    expect = np.sort(np.r_[np.ones(K - 1), 1.0 - np.sum(b * k * k)])
    np.testing.assert_allclose(ev, expect, atol=1e-10)


def test_qed_difference_identities_and_gdn2():
    """QED notes, sec. 2.3, Eqs. 11-12: against GDN-2 on the same Sbar,
    S_QED - S_GDN2 = -lambda k (Sbar^T d)^T and o_QED - o_GDN2 = -lambda rho Sbar^T d,
    with per-channel decay in play; lambda_h = 0 is the GDN-2 update of Eqs. 4/8."""
    K, V = 6, 5
    k = _unit(rng.standard_normal(K))
    q = _unit(rng.standard_normal(K))
    b = rng.uniform(0.05, 0.95, K)
    w = rng.uniform(0.05, 0.95, V)
    v = rng.standard_normal(V)
    g = -rng.uniform(0.0, 0.5, K)
    S_prev = rng.standard_normal((K, V))
    lam = 0.37
    S_q, o_q = _qed_one_step(k, q, b, S_prev, w, v, lam, g)
    S_g, o_g = _qed_one_step(k, q, b, S_prev, w, v, 0.0, g)
    Sbar = np.exp(g)[:, None] * S_prev
    # GDN-2 written from its own equations (the base erase vector b*k)
    r_base = w * v - Sbar.T @ (b * k)
    np.testing.assert_allclose(S_g, Sbar + np.outer(k, r_base), atol=1e-13)
    u = b * q
    d = u - k * np.dot(k, u)
    assert abs(np.dot(d, k)) < 1e-14                       # d is orthogonal to k
    np.testing.assert_allclose(S_q - S_g, -lam * np.outer(k, Sbar.T @ d), atol=1e-13)
    np.testing.assert_allclose(o_q - o_g, -lam * np.dot(q, k) * (Sbar.T @ d), atol=1e-13)


def test_qed_key_orthogonal_response_and_gdn2_decomposition():
    """QED notes, sec. 2.3: Eq. 9 (a probe x orthogonal to k sees no change:
    S_t^T x = Sbar^T x) and Eq. 10 (GDN-2 output split along k and q_perp)."""
    K, V = 7, 4
    k = _unit(rng.standard_normal(K))
    q = _unit(rng.standard_normal(K))
    b = rng.uniform(0.05, 0.95, K)
    w = rng.uniform(0.05, 0.95, V)
    v = rng.standard_normal(V)
    S_prev = rng.standard_normal((K, V))
    for lam in (0.0, 0.8):
        S, o = _qed_one_step(k, q, b, S_prev, w, v, lam)
        x = rng.standard_normal(K)
        x -= k * np.dot(k, x)
        np.testing.assert_allclose(S.T @ x, S_prev.T @ x, atol=1e-13)
    S, o = _qed_one_step(k, q, b, S_prev, w, v, 0.0)
    rho = np.dot(q, k)
    q_perp = q - rho * k
    expect = rho * (w * v + S_prev.T @ ((1.0 - b) * k)) + S_prev.T @ q_perp
    np.testing.assert_allclose(o, expect, atol=1e-13)


def test_qed_decay_only():
    """With v = 0 and b = 0 (nothing erased, nothing written), each key row of the
    state decays by exp(sum of its g) and o = S^T q."""
    K, V, T = 5, 3, 6
    S0 = rng.standard_normal((1, 1, V, K))
    g = -rng.uniform(0, 0.3, (1, T, 1, K))
    q = rng.standard_normal((1, T, 1, K))
    k = _unit(rng.standard_normal((1, T, 1, K)))
    z = np.zeros((1, T, 1, K))
    o, S = oracle.qed_fwd(q, k, np.zeros((1, T, 1, V)), g, z, np.ones((1, T, 1, V)),
                          np.array([0.7]), S0)
    np.testing.assert_allclose(S[0, 0], S0[0, 0] * np.exp(g.sum(axis=1))[0, 0][None, :], atol=1e-14)


# ------------------------------------------ QED ablation arms and decode (page 3)

def _qed_variant_step(k, q, b, S_prev_KxV, w, v, lam_h, variant, z=None, g=None):
    """One oracle step of a QED ablation arm from S0 = S_prev. Returns (S_KxV, o)."""
    K, V = S_prev_KxV.shape
    sh = lambda x: np.asarray(x, dtype=np.float64).reshape(1, 1, 1, -1)
    g = np.zeros(K) if g is None else g
    S0 = S_prev_KxV.T.reshape(1, 1, V, K)
    zz = None if z is None else np.asarray(z, dtype=np.float64).reshape(1, K)
    o, S = oracle.qed_fwd_variant(sh(q), sh(k), sh(v), sh(g), sh(b), sh(w), np.array([lam_h]), variant, zz, S0)
    return S[0, 0].T, o[0, 0, 0]


@pytest.mark.parametrize("variant,z,S_first,o", [
    # the new erase term of each arm (QED notes, sec. 3.2, Table 1) on the sec. 2.4
    # example, k=(1,0), q=(0.6,0.8), b=(0.5,0.5), Sbar=(2,3), w*v=1, lambda=0.2:
    #   full:          d = P(b*q) = (0,0.4),  Sbar^T d = 1.2,  S_1 = 2 - 0.2*1.2 = 1.76
    #   nogate:        d = P(q)   = (0,0.8),  Sbar^T d = 2.4,  S_1 = 2 - 0.48     = 1.52
    #   nogate-noproj: a = b*k + 0.2 q = (0.62,0.16), r = 1 - (1.24+0.48) = -0.72,
    #                  S_1 = 2 - 0.72 = 1.28
    #   rand, z=(0,1): d = P(b*z) = (0,0.5),  Sbar^T d = 1.5,  S_1 = 2 - 0.3      = 1.70
    # and o = 0.6 S_1 + 0.8 * 3 (the second coordinate never changes)
    ("full", None, 1.76, 3.456),
    ("nogate", None, 1.52, 3.312),
    ("nogate_noproj", None, 1.28, 3.168),
    ("rand", [0.0, 1.0], 1.70, 3.42),
])
def test_qed_ablation_arms_on_the_2d_example(variant, z, S_first, o):
    S, out = _qed_variant_step([1.0, 0.0], [0.6, 0.8], [0.5, 0.5], np.array([[2.0], [3.0]]), [1.0], [1.0],
                               0.2, variant, z)
    np.testing.assert_allclose(S.ravel(), [S_first, 3.0], atol=1e-14)
    assert abs(out - o) < 1e-14
    assert abs(out - (0.6 * S_first + 2.4)) < 1e-14


@pytest.mark.parametrize("variant", ["full", "nogate", "nogate_noproj", "rand"])
def test_qed_ablation_arms_difference_identity(variant):
    """QED notes, Eqs. 11-12 hold for every arm with its own new term t
    (S_arm - S_GDN2 = -lambda k (Sbar^T t)^T, o_arm - o_GDN2 = -lambda rho Sbar^T t),
    and the projected arms keep the erase factor's eigenvalue 1 - (b*k)^T k."""
    K, V = 6, 5
    k = _unit(rng.standard_normal(K))
    q = _unit(rng.standard_normal(K))
    z = _unit(rng.standard_normal(K))
    b = rng.uniform(0.05, 0.95, K)
    w = rng.uniform(0.05, 0.95, V)
    v = rng.standard_normal(V)
    g = -rng.uniform(0.0, 0.5, K)
    S_prev = rng.standard_normal((K, V))
    lam = 0.41
    S_a, o_a = _qed_variant_step(k, q, b, S_prev, w, v, lam, variant, z, g)
    S_g, o_g = _qed_variant_step(k, q, b, S_prev, w, v, 0.0, "full", None, g)
    P = lambda u: u - k * np.dot(k, u)
    t = {"full": P(b * q), "nogate": P(q), "nogate_noproj": q, "rand": P(b * z)}[variant]
    Sbar = np.exp(g)[:, None] * S_prev
    np.testing.assert_allclose(S_a - S_g, -lam * np.outer(k, Sbar.T @ t), atol=1e-13)
    np.testing.assert_allclose(o_a - o_g, -lam * np.dot(q, k) * (Sbar.T @ t), atol=1e-13)
    # erase factor M = I - k a^T read off with v = 0, S0 = I, g = 0
    M, _ = _qed_variant_step(k, q, b, np.eye(K), np.ones(K), np.zeros(K), lam, variant, z)
    ev = np.sort(np.linalg.eigvals(M).real)
    shift = 0.0 if variant != "nogate_noproj" else lam * np.dot(k, q)
    expect = np.sort(np.r_[np.ones(K - 1), 1.0 - np.sum(b * k * k) - shift])
    np.testing.assert_allclose(ev, expect, atol=1e-10)


def test_qed_ablation_arms_coincide_where_they_should():
    """b = 1 makes full and nogate the same arm; q orthogonal to k makes nogate and
    nogate-noproj the same; z_h equal to every token's q makes rand and full the same."""
    B, T, H, K, V = 1, 12, 2, 6, 4
    q = _unit(rng.standard_normal((B, T, H, K)))
    k = _unit(rng.standard_normal((B, T, H, K)))
    v = rng.standard_normal((B, T, H, V))
    g = -rng.uniform(0.0, 0.2, (B, T, H, K))
    b = rng.uniform(0.05, 0.95, (B, T, H, K))
    w = rng.uniform(0.05, 0.95, (B, T, H, V))
    lam = np.array([0.3, 0.9])
    S0 = rng.standard_normal((B, H, V, K)) * 0.3
    ones = np.ones_like(b)
    o1, S1 = oracle.qed_fwd_variant(q, k, v, g, ones, w, lam, "full", None, S0)
    o2, S2 = oracle.qed_fwd_variant(q, k, v, g, ones, w, lam, "nogate", None, S0)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(S1, S2)
    q_perp = _unit(q - k * np.sum(k * q, axis=-1, keepdims=True))
    o1, S1 = oracle.qed_fwd_variant(q_perp, k, v, g, b, w, lam, "nogate", None, S0)
    o2, S2 = oracle.qed_fwd_variant(q_perp, k, v, g, b, w, lam, "nogate_noproj", None, S0)
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    np.testing.assert_allclose(S1, S2, atol=1e-12)
    zh = _unit(rng.standard_normal((H, K)))
    q_const = np.broadcast_to(zh[None, None], (B, T, H, K)).copy()
    o1, S1 = oracle.qed_fwd_variant(q_const, k, v, g, b, w, lam, "full", None, S0)
    o2, S2 = oracle.qed_fwd_variant(q_const, k, v, g, b, w, lam, "rand", zh, S0)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(S1, S2)
    # the full arm through the variant entry point is the QED forward itself
    o1, S1 = oracle.qed_fwd_variant(q, k, v, g, b, w, lam, "full", None, S0)
    o2, S2 = oracle.qed_fwd(q, k, v, g, b, w, lam, S0)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(S1, S2)


@pytest.mark.parametrize("variant", ["full", "nogate_noproj", "rand"])
def test_qed_step_sequence_equals_forward(variant):
    """T decode steps carry the state exactly as one forward over the T tokens."""
    N, T, H, K, V = 2, 5, 3, 6, 4
    q = _unit(rng.standard_normal((N, T, H, K)))
    k = _unit(rng.standard_normal((N, T, H, K)))
    v = rng.standard_normal((N, T, H, V))
    g = -rng.uniform(0.0, 0.2, (N, T, H, K))
    b = rng.uniform(0.05, 0.95, (N, T, H, K))
    w = rng.uniform(0.05, 0.95, (N, T, H, V))
    lam = rng.uniform(0.0, 1.0, H)
    z = _unit(rng.standard_normal((H, K)))
    S0 = rng.standard_normal((N, H, V, K)) * 0.3
    o_f, S_f = oracle.qed_fwd_variant(q, k, v, g, b, w, lam, variant, z, S0)
    S = S0.copy()
    for t in range(T):
        o_t = oracle.qed_step(S, q[:, t], k[:, t], v[:, t], g[:, t], b[:, t], w[:, t], lam, variant, z)
        np.testing.assert_array_equal(o_t, o_f[:, t])
    np.testing.assert_array_equal(S, S_f)


# ------------------------------------------------ prologue (DeltaNet 3.8, Q-Delta 2.5)

def _plain_vs_prologue(q_raw, k_raw, q, k, a_logit, alpha, b_logit, beta, l_logit, lam, atol):
    """The prologue forward on raw inputs equals the plain forward on the feature map's
    and gates' closed-form values."""
    T, H, d = q_raw.shape[1:]
    v = rng.standard_normal((1, T, H, d))
    S0 = rng.standard_normal((1, H, d, d)) * 0.3
    o1, S1 = oracle.qdelta_fwd_prologue(q_raw, k_raw, v, a_logit, b_logit, l_logit, S0)
    o2, S2 = oracle.qdelta_fwd(q, k, v, alpha, beta, lam, S0)
    np.testing.assert_allclose(o1, o2, atol=atol)
    np.testing.assert_allclose(S1, S2, atol=atol)


def test_prologue_silu_shape_and_l2_norm():
    """SiLU(x) = x sigmoid(x): sigmoid(ln 3) = 3/4 and sigmoid(-ln 3) = 1/4, so the raw row
    (ln 3, -ln 3) maps to (3 ln3/4, -ln3/4) / |.| = (3, -1)/sqrt(10); a zero entry stays 0."""
    T, H = 4, 2
    l3 = np.log(3.0)
    row = np.array([l3, -l3, 0.0, 0.0])
    q_raw = np.broadcast_to(row, (1, T, H, 4)).copy()
    k_raw = np.broadcast_to(row[[2, 0, 3, 1]], (1, T, H, 4)).copy()
    q = np.broadcast_to(np.array([3.0, -1.0, 0.0, 0.0]) / np.sqrt(10.0), (1, T, H, 4)).copy()
    k = np.broadcast_to(np.array([0.0, 3.0, 0.0, -1.0]) / np.sqrt(10.0), (1, T, H, 4)).copy()
    z = np.zeros((1, T, H))
    # logit 0: sigmoid(0) = 1/2 and exp(-softplus(0)) = exp(-ln 2) = 1/2
    half = np.full((1, T, H), 0.5)
    _plain_vs_prologue(q_raw, k_raw, q, k, z, half, z, half, z, half, atol=1e-14)


def test_prologue_gates_closed_forms():
    """exp(-softplus(x)) = 1/(1 + e^x) and sigmoid(x) = 1/(1 + e^-x) for the gate logits,
    with one-hot features (one large entry, the others far negative: SiLU ~ 0)."""
    T, H, d = 6, 3, 5
    q_raw = np.full((1, T, H, d), -60.0)
    k_raw = np.full((1, T, H, d), -60.0)
    idx_q = rng.integers(0, d, (T, H))
    idx_k = rng.integers(0, d, (T, H))
    q = np.zeros((1, T, H, d))
    k = np.zeros((1, T, H, d))
    for t in range(T):
        for h in range(H):
            q_raw[0, t, h, idx_q[t, h]] = 2.5
            k_raw[0, t, h, idx_k[t, h]] = 4.0
            q[0, t, h, idx_q[t, h]] = 1.0
            k[0, t, h, idx_k[t, h]] = 1.0
    a_l, b_l, l_l = [rng.uniform(-4, 4, (1, T, H)) for _ in range(3)]
    alpha = 1.0 / (1.0 + np.exp(a_l))
    beta = 1.0 / (1.0 + np.exp(-b_l))
    lam = 1.0 / (1.0 + np.exp(-l_l))
    _plain_vs_prologue(q_raw, k_raw, q, k, a_l, alpha, b_l, beta, l_l, lam, atol=1e-12)
    # absent alpha / lambda logits: alpha = 1, lambda = 0
    _plain_vs_prologue(q_raw, k_raw, q, k, None, None, b_l, beta, None, None, atol=1e-12)


def test_prologue_large_inputs_reduce_to_l2_normalisation():
    """For large positive entries SiLU(x) = x (to 1e-17), so the feature map is x/|x|."""
    T, H, d = 5, 2, 6
    u = rng.uniform(1.0, 2.0, (1, T, H, d))
    w = rng.uniform(1.0, 2.0, (1, T, H, d))
    _plain_vs_prologue(60.0 * u, 60.0 * w, u / np.linalg.norm(u, axis=-1, keepdims=True),
                       w / np.linalg.norm(w, axis=-1, keepdims=True), None, None,
                       np.zeros((1, T, H)), np.full((1, T, H), 0.5), None, None, atol=1e-12)


# ------------------------------------------------------------ Q-Delta (page 1)

def test_deltanet_special_case():
    """lambda = 0, alpha = 1 is DeltaNet: compared with the DeltaNet notes' own
    read / blend / replace form (sec. 2.5): v_old = S k, v_new = beta v + (1-beta) v_old,
    S <- S - v_old k^T + v_new k^T."""
    q, k, v, _, beta, _, S0 = _rand_qdelta(1, 12, 1, 6, 5, gated=False, lam=False)
    o, S = oracle.qdelta_fwd(q, k, v, None, beta, None, S0)
    St = S0[0, 0].copy()
    for t in range(12):
        kt, vt, bt = k[0, t, 0], v[0, t, 0], beta[0, t, 0]
        v_old = St @ kt
        v_new = bt * vt + (1 - bt) * v_old
        St = St - np.outer(v_old, kt) + np.outer(v_new, kt)
        np.testing.assert_allclose(o[0, t, 0], St @ q[0, t, 0], atol=1e-12)
    np.testing.assert_allclose(S[0, 0], St, atol=1e-12)


def test_gated_deltanet_special_case():
    """lambda = 0 is Gated DeltaNet: S_t = S_{t-1} alpha_t (I - beta_t k k^T) + beta_t v k^T
    (DeltaNet notes sec. 6.2), as explicit matrix products."""
    q, k, v, alpha, beta, _, S0 = _rand_qdelta(1, 10, 1, 5, 4, lam=False)
    o, S = oracle.qdelta_fwd(q, k, v, alpha, beta, None, S0)
    St = S0[0, 0].copy()
    I = np.eye(5)
    for t in range(10):
        kt, vt = k[0, t, 0], v[0, t, 0]
        St = St @ (alpha[0, t, 0] * (I - beta[0, t, 0] * np.outer(kt, kt))) + beta[0, t, 0] * np.outer(vt, kt)
        np.testing.assert_allclose(o[0, t, 0], St @ q[0, t, 0], atol=1e-12)
    np.testing.assert_allclose(S[0, 0], St, atol=1e-12)


def test_beta_zero_pure_decay():
    """beta = 0: nothing is written, S_T = (prod alpha) S_0 and o_t = gamma_t S_0 q_t."""
    q, k, v, alpha, beta, lam, S0 = _rand_qdelta(2, 9, 3, 6, 4)
    beta = np.zeros_like(beta)
    o, S = oracle.qdelta_fwd(q, k, v, alpha, beta, lam, S0)
    gam = np.cumprod(alpha, axis=1)                      # [B,T,H]
    np.testing.assert_allclose(S, S0 * gam[:, -1][:, :, None, None], atol=1e-13)
    expect = np.einsum("bth,bhij,bthj->bthi", gam, S0, q)
    np.testing.assert_allclose(o, expect, atol=1e-13)
    o0, S00 = oracle.qdelta_fwd(q, k, v, alpha, beta, lam, None)
    assert np.all(o0 == 0) and np.all(S00 == 0)          # beta = 0 from S_0 = 0 stays 0


def test_exact_retrieval_orthonormal_keys():
    """beta = 1, alpha = 1, lambda = 0 with orthonormal keys: S k_j = v_j for every
    key written (DeltaNet notes sec. 2.5: beta = 1 replaces the value)."""
    d, dv = 8, 5
    Qm, _ = np.linalg.qr(rng.standard_normal((d, d)))
    k = Qm.T.reshape(1, d, 1, d)
    v = rng.standard_normal((1, d, 1, dv))
    q = _unit(rng.standard_normal((1, d, 1, d)))
    beta = np.ones((1, d, 1))
    S0 = rng.standard_normal((1, 1, dv, d))
    _, S = oracle.qdelta_fwd(q, k, v, None, beta, None, S0)
    np.testing.assert_allclose(S[0, 0] @ k[0, :, 0].T, v[0, :, 0].T, atol=1e-12)


def test_exact_write_beta_inverse_norm():
    """DeltaNet notes sec. 2.6: with beta = 1/|k|^2 one step gives S_t k_t = v_t."""
    d, dv = 6, 4
    k = rng.standard_normal((1, 1, 1, d)) * 1.7
    v = rng.standard_normal((1, 1, 1, dv))
    q = rng.standard_normal((1, 1, 1, d))
    beta = np.array([[[1.0 / np.sum(k ** 2)]]])
    _, S = oracle.qdelta_fwd(q, k, v, None, beta, None, rng.standard_normal((1, 1, dv, d)))
    np.testing.assert_allclose(S[0, 0] @ k[0, 0, 0], v[0, 0, 0], atol=1e-12)


def test_deltanet_transition_eigenvalues():
    """DeltaNet notes sec. 3.8: I - beta k k^T has eigenvalue 1 (d-1 times) and
    1 - beta |k|^2.  Read off the oracle with v = 0 and S_0 = I."""
    d = 6
    k = rng.standard_normal((1, 1, 1, d))
    beta = np.array([[[0.6]]])
    _, S = oracle.qdelta_fwd(np.zeros((1, 1, 1, d)), k, np.zeros((1, 1, 1, d)), None, beta,
                             None, np.eye(d).reshape(1, 1, d, d))
    ev = np.sort(np.linalg.eigvals(S[0, 0]).real)
    expect = np.sort(np.r_[np.ones(d - 1), 1 - 0.6 * np.sum(k ** 2)])
    np.testing.assert_allclose(ev, expect, atol=1e-12)


def _value_mixture(q, k, v, alpha, beta, lam, S0):
    """Q-Delta notes sec. 2.2 (Eqs. 8-15): for S_t = S_{t-1} P_t + eta_t v_t k_t^T,
    S_t = S_0 P_1..P_t + sum_tau v_tau b_{tau,t}^T with b_{tau,t} = P_t^T b_{tau,t-1},
    b_{tau,tau} = eta_tau k_tau.  Here P_t = alpha_t (I - beta_t x_t k_t^T), eta = beta."""
    T, dk = q.shape[1], q.shape[-1]
    I = np.eye(dk)
    P = []
    for t in range(T):
        x = k[0, t, 0] + lam[0, t, 0] * q[0, t, 0]
        P.append(alpha[0, t, 0] * (I - beta[0, t, 0] * np.outer(x, k[0, t, 0])))
    outs, S_list = [], []
    for t in range(T):
        prod = I.copy()
        for j in range(t + 1):
            prod = prod @ P[j]
        St = S0[0, 0] @ prod
        for tau in range(t + 1):
            bvec = beta[0, tau, 0] * k[0, tau, 0]
            for j in range(tau + 1, t + 1):
                bvec = P[j].T @ bvec
            St = St + np.outer(v[0, tau, 0], bvec)
        S_list.append(St)
        outs.append(St @ q[0, t, 0])
    return outs, S_list


@pytest.mark.parametrize("T", [1, 2, 5, 8])
def test_value_mixture_bruteforce(T):
    q, k, v, alpha, beta, lam, S0 = _rand_qdelta(1, T, 1, 5, 4)
    o, S = oracle.qdelta_fwd(q, k, v, alpha, beta, lam, S0)
    outs, S_list = _value_mixture(q, k, v, alpha, beta, lam, S0)
    for t in range(T):
        np.testing.assert_allclose(o[0, t, 0], outs[t], atol=1e-12)
    np.testing.assert_allclose(S[0, 0], S_list[-1], atol=1e-12)


def test_gated_error_identity_and_closed_form_output():
    """Q-Delta notes sec. 2.7 (gated): v_t - S_t x_t = (1 - beta_t a_t)(v_t - alpha_t S_{t-1} x_t),
    a_t = k_t^T x_t; sec. 2.4: o_t = alpha S_{t-1} q + beta (v - alpha S_{t-1} x)(k^T q)."""
    q, k, v, alpha, beta, lam, S0 = _rand_qdelta(1, 10, 1, 6, 5)
    states, outs = _states_per_step(q, k, v, alpha, beta, lam, S0)
    for t in range(10):
        qt, kt, vt = q[0, t, 0], k[0, t, 0], v[0, t, 0]
        al, be, lm = alpha[0, t, 0], beta[0, t, 0], lam[0, t, 0]
        x = kt + lm * qt
        Sp, S = states[t], states[t + 1]
        a = kt @ x
        np.testing.assert_allclose(vt - S @ x, (1 - be * a) * (vt - al * Sp @ x), atol=1e-12)
        o_cf = al * Sp @ qt + be * (vt - al * Sp @ x) * (kt @ qt)
        np.testing.assert_allclose(outs[t], o_cf, atol=1e-12)


def test_lemma31_ungated_contraction():
    """Q-Delta notes sec. 2.7, Lemma 3.1 (alpha = 1): e_t = (1 - beta_t a_t) e~_t with
    e~_t = v_t - S_{t-1} x_t; for unit q, k also 1 - lambda <= a_t <= 1 + lambda."""
    q, k, v, _, beta, lam, S0 = _rand_qdelta(1, 10, 1, 6, 5, gated=False)
    states, _ = _states_per_step(q, k, v, None, beta, lam, S0)
    for t in range(10):
        x = k[0, t, 0] + lam[0, t, 0] * q[0, t, 0]
        a = k[0, t, 0] @ x
        e_tilde = v[0, t, 0] - states[t] @ x
        e = v[0, t, 0] - states[t + 1] @ x
        np.testing.assert_allclose(e, (1 - beta[0, t, 0] * a) * e_tilde, atol=1e-12)
        assert 1 - lam[0, t, 0] - 1e-12 <= a <= 1 + lam[0, t, 0] + 1e-12


def test_online_surrogate_minimiser():
    """Q-Delta notes sec. 2.5 (Table 1): the minimiser of
    J(S) = |S - alpha S_{t-1}|_F^2 - 2 beta <S k, delta>, delta = v - alpha S_{t-1} x,
    found by a generic least-squares solve of the quadratic, is the oracle's step."""
    dk, dv = 4, 3
    q, k, v, alpha, beta, lam, S0 = _rand_qdelta(1, 1, 1, dk, dv)
    _, S1 = oracle.qdelta_fwd(q, k, v, alpha, beta, lam, S0)
    Sp = S0[0, 0]
    al, be = alpha[0, 0, 0], beta[0, 0, 0]
    x = k[0, 0, 0] + lam[0, 0, 0] * q[0, 0, 0]
    delta = v[0, 0, 0] - al * Sp @ x
    # J(s) = s^T s - 2 s^T (alpha vec(Sp)) - 2 beta s^T (delta kron k) + const  (s = vec(S), row-major)
    # as least squares: min |s - c|^2 with c the stationary point of the linear terms
    n = dv * dk
    A = np.eye(n)
    lin = al * Sp.reshape(-1) + be * np.array([delta[i] * k[0, 0, 0][j] for i in range(dv) for j in range(dk)])
    s, *_ = np.linalg.lstsq(A, lin, rcond=None)
    # independent check that s is the minimiser: J increases along random directions
    J = lambda S: np.sum((S - al * Sp) ** 2) - 2 * be * np.dot(S @ k[0, 0, 0], delta)
    Smin = s.reshape(dv, dk)
    for _ in range(5):
        D = rng.standard_normal((dv, dk)) * 1e-3
        assert J(Smin + D) > J(Smin) and J(Smin - D) > J(Smin)
    np.testing.assert_allclose(S1[0, 0], Smin, atol=1e-12)


# -------------------------------------------------- equivalences of the oracle

def test_step_equals_forward():
    q, k, v, alpha, beta, lam, S0 = _rand_qdelta(3, 7, 2, 6, 5)
    o, S = oracle.qdelta_fwd(q, k, v, alpha, beta, lam, S0)
    St = S0.copy()
    for t in range(7):
        ot = oracle.qdelta_step(St, q[:, t], k[:, t], v[:, t], alpha[:, t], beta[:, t], lam[:, t])
        np.testing.assert_allclose(ot, o[:, t], atol=1e-12)
    np.testing.assert_allclose(St, S, atol=1e-12)


@pytest.mark.parametrize("split", [1, 5, 11])
def test_split_call_carries_state(split):
    q, k, v, alpha, beta, lam, S0 = _rand_qdelta(2, 12, 2, 5, 4)
    o, S = oracle.qdelta_fwd(q, k, v, alpha, beta, lam, S0)
    a = slice(0, split)
    b = slice(split, 12)
    o1, S1 = oracle.qdelta_fwd(q[:, a], k[:, a], v[:, a], alpha[:, a], beta[:, a], lam[:, a], S0)
    o2, S2 = oracle.qdelta_fwd(q[:, b], k[:, b], v[:, b], alpha[:, b], beta[:, b], lam[:, b], S1)
    np.testing.assert_allclose(np.concatenate([o1, o2], axis=1), o, atol=1e-12)
    np.testing.assert_allclose(S2, S, atol=1e-12)


def test_heads_and_batches_independent_and_thread_count_invariant():
    q, k, v, alpha, beta, lam, S0 = _rand_qdelta(3, 6, 4, 5, 3)
    o, S = oracle.qdelta_fwd(q, k, v, alpha, beta, lam, S0, nthreads=1)
    o4, S4 = oracle.qdelta_fwd(q, k, v, alpha, beta, lam, S0, nthreads=5)
    assert np.array_equal(o, o4) and np.array_equal(S, S4)
    b, h = 2, 1
    sl = lambda x: x[b:b + 1, :, h:h + 1]
    o1, S1 = oracle.qdelta_fwd(sl(q), sl(k), sl(v), sl(alpha), sl(beta), sl(lam), S0[b:b + 1, h:h + 1])
    assert np.array_equal(o1[0, :, 0], o[b, :, h]) and np.array_equal(S1[0, 0], S[b, h])


# ---------------------------------------------------------------- backward

def _loss(q, k, v, alpha, beta, lam, S0, dO, dS):
    o, S = oracle.qdelta_fwd(q, k, v, alpha, beta, lam, S0)
    return float((o * dO).sum() + (S * dS).sum())


def finite_difference_grads(q, k, v, alpha, beta, lam, S0, dO, dS, h=1e-6):
    """Central differences of L = <dO, o> + <dS, S_T> through the (pinned) forward
    oracle, for every element of every input."""
    args = {"q": q, "k": k, "v": v, "alpha": alpha, "beta": beta, "lam": lam, "S0": S0}
    out = {}
    for name, x in args.items():
        if x is None:
            continue
        fd = np.zeros_like(x)
        for i in np.ndindex(x.shape):
            a = dict(args)
            xp, xm = x.copy(), x.copy()
            xp[i] += h
            xm[i] -= h
            a[name] = xp
            lp = _loss(**a, dO=dO, dS=dS)
            a[name] = xm
            lm = _loss(**a, dO=dO, dS=dS)
            fd[i] = (lp - lm) / (2 * h)
        out["d" + name] = fd
    return out


@pytest.mark.parametrize("mode", ["qdelta", "gdn", "deltanet"])
def test_backward_equals_finite_differences(mode):
    """Every gradient of the backward oracle is the derivative of the forward oracle
    (central differences, h = 1e-6; truncation ~1e-12, cancellation ~1e-10)."""
    q, k, v, alpha, beta, lam, S0 = _rand_qdelta(1, 7, 2, 4, 3, gated=mode != "deltanet", lam=mode == "qdelta",
                                                 unit=False)
    alpha = None if alpha is None else rng.uniform(0.5, 1.0, alpha.shape)
    dO = rng.standard_normal(v.shape)
    dS = rng.standard_normal(S0.shape)
    g = oracle.qdelta_bwd(q, k, v, alpha, beta, lam, S0, dO, dS)
    fd = finite_difference_grads(q, k, v, alpha, beta, lam, S0, dO, dS)
    for name, ref in fd.items():
        np.testing.assert_allclose(g[name], ref, atol=1e-6 * max(1.0, np.abs(ref).max()), err_msg=name)
    assert (g["dalpha"] is None) == (alpha is None) and (g["dlam"] is None) == (lam is None)


def test_backward_linear_in_values_and_initial_state():
    """o and S_T are jointly linear in (v, S0) (each step is S_prior (I - beta x k^T)
    + beta v k^T), so by Euler's identity <dv, v> + <dS0, S0> = L exactly."""
    q, k, v, alpha, beta, lam, S0 = _rand_qdelta(2, 23, 3, 8, 6)
    dO, dS = rng.standard_normal(v.shape), rng.standard_normal(S0.shape)
    g = oracle.qdelta_bwd(q, k, v, alpha, beta, lam, S0, dO, dS)
    L = _loss(q, k, v, alpha, beta, lam, S0, dO, dS)
    assert abs((g["dv"] * v).sum() + (g["dS0"] * S0).sum() - L) <= 1e-11 * max(1.0, abs(L))


def test_backward_linear_in_queries_without_lambda():
    """lambda = 0: the states do not depend on q and o_t = S_t q_t is linear in it,
    so <dq, q> = <dO, o> (with lambda != 0 the identity fails, as x carries q)."""
    q, k, v, alpha, beta, _, S0 = _rand_qdelta(2, 17, 2, 8, 5, lam=False)
    dO = rng.standard_normal(v.shape)
    o, _ = oracle.qdelta_fwd(q, k, v, alpha, beta, None, S0)
    g = oracle.qdelta_bwd(q, k, v, alpha, beta, None, S0, dO)
    ref = (dO * o).sum()
    assert abs((g["dq"] * q).sum() - ref) <= 1e-12 * max(1.0, abs(ref))
    lam = rng.uniform(0.2, 0.8, beta.shape)
    o2, _ = oracle.qdelta_fwd(q, k, v, alpha, beta, lam, S0)
    g2 = oracle.qdelta_bwd(q, k, v, alpha, beta, lam, S0, dO)
    assert abs((g2["dq"] * q).sum() - (dO * o2).sum()) > 1e-6


def test_backward_beta_zero_closed_form():
    """beta = 0: S_t = gamma_t S0.  The gradient reaching S_t is
    G_t = sum_{tau>=t} (gamma_tau/gamma_t) dO_tau q_tau^T + (gamma_T/gamma_t) dS_T, so
    dbeta_t = e_t^T G_t k_t with e_t = v_t - gamma_t S0 x_t; dq_t = gamma_t S0^T dO_t;
    dk = dv = dlambda = 0; alpha_j dalpha_j = sum_{t>=j} gamma_t <dO_t, S0 q_t>
    + gamma_T <dS_T, S0>; dS0 = sum_t gamma_t dO_t q_t^T + gamma_T dS_T."""
    B, T, H, dk, dv = 1, 9, 2, 5, 4
    q, k, v, alpha, beta, lam, S0 = _rand_qdelta(B, T, H, dk, dv)
    beta = np.zeros_like(beta)
    dO, dS = rng.standard_normal(v.shape), rng.standard_normal(S0.shape)
    g = oracle.qdelta_bwd(q, k, v, alpha, beta, lam, S0, dO, dS)
    for h in range(H):
        gam = np.cumprod(alpha[0, :, h])
        S0h, dSh = S0[0, h], dS[0, h]
        Q, K, V, dOh = q[0, :, h], k[0, :, h], v[0, :, h], dO[0, :, h]
        X = K + lam[0, :, h, None] * Q
        for t in range(T):
            G = sum(gam[u] / gam[t] * np.outer(dOh[u], Q[u]) for u in range(t, T)) + gam[-1] / gam[t] * dSh
            e = V[t] - gam[t] * S0h @ X[t]
            assert abs(g["dbeta"][0, t, h] - e @ G @ K[t]) <= 1e-12 * max(1.0, abs(e @ G @ K[t]))
            np.testing.assert_allclose(g["dq"][0, t, h], gam[t] * S0h.T @ dOh[t], atol=1e-13)
            ref = sum(gam[u] * dOh[u] @ S0h @ Q[u] for u in range(t, T)) + gam[-1] * (dSh * S0h).sum()
            assert abs(alpha[0, t, h] * g["dalpha"][0, t, h] - ref) <= 1e-12 * max(1.0, abs(ref))
        dS0 = sum(gam[u] * np.outer(dOh[u], Q[u]) for u in range(T)) + gam[-1] * dSh
        np.testing.assert_allclose(g["dS0"][0, h], dS0, atol=1e-13)
    assert np.all(g["dk"] == 0) and np.all(g["dv"] == 0) and np.all(g["dlam"] == 0)


def test_backward_streams_independent_and_thread_count_invariant():
    q, k, v, alpha, beta, lam, S0 = _rand_qdelta(2, 11, 3, 6, 5)
    dO, dS = rng.standard_normal(v.shape), rng.standard_normal(S0.shape)
    g1 = oracle.qdelta_bwd(q, k, v, alpha, beta, lam, S0, dO, dS, nthreads=1)
    g4 = oracle.qdelta_bwd(q, k, v, alpha, beta, lam, S0, dO, dS, nthreads=4)
    one = oracle.qdelta_bwd(q[1:, :, 2:], k[1:, :, 2:], v[1:, :, 2:], alpha[1:, :, 2:], beta[1:, :, 2:],
                            lam[1:, :, 2:], S0[1:, 2:], dO[1:, :, 2:], dS[1:, 2:])
    for name in g1:
        assert np.array_equal(g1[name], g4[name]), name
    np.testing.assert_array_equal(one["dq"], g1["dq"][1:, :, 2:])
    np.testing.assert_array_equal(one["dS0"], g1["dS0"][1:, 2:])


# ---------------------------------------------------------------- EDA (erase-then-delta)

def _rand_eda(B, T, H, dk, dv, beta=True):
    q = _unit(rng.standard_normal((B, T, H, dk)))
    k = _unit(rng.standard_normal((B, T, H, dk)))
    e = _unit(rng.standard_normal((B, T, H, dk)))
    v = rng.standard_normal((B, T, H, dv))
    bt = rng.uniform(0.1, 1.0, (B, T, H)) if beta else None
    S0 = rng.standard_normal((B, H, dv, dk)) * 0.3
    return q, k, v, e, bt, S0


def test_eda_erase_along_the_key_is_deltanet():
    """e_t = k_t with unit keys: (I - k k^T)^2 = I - k k^T, so the erase adds nothing to
    the Delta write and EDA with unit step is DeltaNet with beta = 1 (the page's two
    steps then coincide with the standard Delta update it starts from)."""
    q, k, v, _, _, S0 = _rand_eda(2, 13, 2, 6, 5, beta=False)
    o, S = oracle.eda_fwd(q, k, v, k, None, S0)
    o2, S2 = oracle.qdelta_fwd(q, k, v, None, np.ones(q.shape[:3]), None, S0)
    np.testing.assert_allclose(o, o2, atol=1e-12)
    np.testing.assert_allclose(S, S2, atol=1e-12)


def test_eda_erase_only_projects_out_the_direction():
    """Zero key and value: only the erase acts.  After one step the memory has no
    component along e (S e = 0, i.e. e^T M = 0) and S = S0 (I - e e^T); with
    orthonormal directions over the steps, S_T = S0 (I - sum_t e_t e_t^T)."""
    d, dv, T = 8, 5, 4
    Q, _ = np.linalg.qr(rng.standard_normal((d, d)))
    e = Q[:, :T].T.reshape(1, T, 1, d)
    z = np.zeros((1, T, 1, d))
    q = _unit(rng.standard_normal((1, T, 1, d)))
    S0 = rng.standard_normal((1, 1, dv, d))
    _, S1 = oracle.eda_fwd(q[:, :1], z[:, :1], np.zeros((1, 1, 1, dv)), e[:, :1], None, S0)
    np.testing.assert_allclose(S1[0, 0] @ e[0, 0, 0], 0.0, atol=1e-13)
    np.testing.assert_allclose(S1[0, 0], S0[0, 0] @ (np.eye(d) - np.outer(e[0, 0, 0], e[0, 0, 0])), atol=1e-13)
    o, ST = oracle.eda_fwd(q, z, np.zeros((1, T, 1, dv)), e, None, S0)
    P = np.eye(d) - sum(np.outer(e[0, t, 0], e[0, t, 0]) for t in range(T))
    np.testing.assert_allclose(ST[0, 0], S0[0, 0] @ P, atol=1e-13)
    np.testing.assert_allclose(o[0, -1, 0], ST[0, 0] @ q[0, -1, 0], atol=1e-13)


def test_eda_unit_write_retrieves_the_value():
    """beta = 1 and a unit key: after the write S_t k_t = v_t exactly, whatever was
    erased before (the Delta write replaces the key's slot)."""
    q, k, v, e, _, S0 = _rand_eda(1, 9, 3, 6, 4, beta=False)
    for t in range(1, 10):
        _, S = oracle.eda_fwd(q[:, :t], k[:, :t], v[:, :t], e[:, :t], None, S0)
        for h in range(3):
            np.testing.assert_allclose(S[0, h] @ k[0, t - 1, h], v[0, t - 1, h], atol=1e-12)


@pytest.mark.parametrize("T", [1, 3, 6])
def test_eda_bruteforce_transition_products(T):
    """S_T = S0 prod_t A_t + sum_t beta_t v_t k_t^T prod_{u>t} A_u with
    A_t = (I - e_t e_t^T)(I - beta_t k_t k_t^T), by explicit matrices, and every
    o_t = S_t q_t."""
    q, k, v, e, bt, S0 = _rand_eda(1, T, 1, 5, 3)
    o, S = oracle.eda_fwd(q, k, v, e, bt, S0)
    I = np.eye(5)
    A = [(I - np.outer(e[0, t, 0], e[0, t, 0])) @ (I - bt[0, t, 0] * np.outer(k[0, t, 0], k[0, t, 0]))
         for t in range(T)]
    St = S0[0, 0].copy()
    for t in range(T):
        St = St @ A[t] + bt[0, t, 0] * np.outer(v[0, t, 0], k[0, t, 0])
        np.testing.assert_allclose(o[0, t, 0], St @ q[0, t, 0], atol=1e-12)
    ref = S0[0, 0].copy()
    for t in range(T):
        ref = ref @ A[t]
    for t in range(T):
        term = bt[0, t, 0] * np.outer(v[0, t, 0], k[0, t, 0])
        for u in range(t + 1, T):
            term = term @ A[u]
        ref = ref + term
    np.testing.assert_allclose(S[0, 0], ref, atol=1e-12)


def _loss_prologue(q_raw, k_raw, v, a_l, b_l, l_l, S0, dO, dS):
    o, S = oracle.qdelta_fwd_prologue(q_raw, k_raw, v, a_l, b_l, l_l, S0)
    return float((o * dO).sum() + (S * dS).sum())


@pytest.mark.parametrize("gates", ["all", "beta_only"])
def test_prologue_backward_equals_finite_differences(gates):
    """The backward from projections is the derivative of the (pinned) prologue forward:
    central differences for every element of q_raw, k_raw, v, the logits and S0."""
    B, T, H, dk, dv = 1, 6, 2, 4, 3
    q_raw, k_raw = rng.standard_normal((B, T, H, dk)), rng.standard_normal((B, T, H, dk))
    v = rng.standard_normal((B, T, H, dv))
    a_l = rng.normal(-1.0, 0.5, (B, T, H)) if gates == "all" else None
    b_l = rng.standard_normal((B, T, H))
    l_l = rng.standard_normal((B, T, H)) if gates == "all" else None
    S0, dS = rng.standard_normal((B, H, dv, dk)) * 0.3, rng.standard_normal((B, H, dv, dk))
    dO = rng.standard_normal((B, T, H, dv))
    g = oracle.qdelta_bwd_prologue(q_raw, k_raw, v, a_l, b_l, l_l, S0, dO, dS)
    args = {"q": q_raw, "k": k_raw, "v": v, "alpha": a_l, "beta": b_l, "lam": l_l, "S0": S0}
    for name, x in args.items():
        if x is None:
            assert g["d" + name] is None
            continue
        fd = np.zeros_like(x)
        for i in np.ndindex(x.shape):
            a = dict(args)
            xp, xm = x.copy(), x.copy()
            xp[i] += 1e-6
            xm[i] -= 1e-6
            a[name] = xp
            lp = _loss_prologue(a["q"], a["k"], a["v"], a["alpha"], a["beta"], a["lam"], a["S0"], dO, dS)
            a[name] = xm
            lm = _loss_prologue(a["q"], a["k"], a["v"], a["alpha"], a["beta"], a["lam"], a["S0"], dO, dS)
            fd[i] = (lp - lm) / 2e-6
        np.testing.assert_allclose(g["d" + name], fd, atol=1e-6 * max(1.0, np.abs(fd).max()), err_msg=name)
